// Grouped GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One persistent, warp-specialised kernel serves four uses:
//   * FP8 expert GEMMs with fine-grained scales (DeepSeek-V3 Technical Report,
//     learn.ifs.name summary, paragraphs on FP8 tiles and on promotion): each
//     128-wide K block is multiplied by the tensor cores into its own TMEM
//     buffer; epilogue warps read it, multiply by sa[row,kb] * sb[nblk,kb]
//     and add it into FP32 registers, while the tensor cores fill the other
//     buffer with the next block.
//   * bf16 expert GEMMs (TMEM partial sums of 8 K steps added into FP32
//     registers).
//   * the gate logits of routing (bf16, split-K partial sums in fp32).
//   * FP8 weight gradients of the layer's backward pass (the groups split K,
//     not M: each expert's tokens are its own K range, padded to 128; both
//     operands carry one scale per (128-token block, row), so each 128-K
//     partial sum is multiplied by sa[row,kb] * sb[col,kb] before it is added
//     into fp32 registers).
//
// Block roles (608 threads):
//   warps 0-15  epilogue: warp w reads TMEM lanes 32*(w%4).. (rows); in
//               warpgroup w/4 it takes the columns {32*(w/4) + c} and
//               {128 + 32*(w/4) + c} of a SwiGLU tile (gate and up side by
//               side), else the 64 contiguous columns {64*(w/4) + c};
//   warp 16     TMA producer: one lane issues the tile loads and does nothing
//               else (any other work in its loop delays the loads);
//   warp 17     tcgen05.mma issuer (one elected lane) + TMEM owner;
//   warp 18     FP8 scales: each K block's 128 row scales and 2 weight scales
//               copied into a shared-memory ring (cp.async), so the epilogue
//               never waits on a global load inside its promotion loop.
// Tile: 128 rows x 256 columns, K step 128 bytes (128 e4m3 or 64 bf16),
// 4-stage shared-memory ring (48 KB per stage), 2 x 256 TMEM columns.
// The SwiGLU FP8 epilogue can also store the tile's fp32 products rounded to
// bf16 (the training forward keeps them for the backward pass).
#include "common.cuh"
#include "gemm.cuh"

namespace moe {

namespace {

constexpr int kStages = 4;   // shared-memory ring depth (the weight gradient's: 2)
constexpr int kBM = 128, kBN = 256;
constexpr int kABytes = kBM * 128, kBBytes = kBN * 128;
constexpr int kEpiWarps = 16, kThreads = (kEpiWarps + 3) * 32;
constexpr int kProducerWarp = kEpiWarps, kMmaWarp = kEpiWarps + 1, kScaleWarp = kEpiWarps + 2;
constexpr int kMaxGroups = 1024;
constexpr int kSSlots = 8;   // K blocks of scales staged ahead of the epilogue

// kSbN: FP8 forward, the weight scales of the tile's two 128-column blocks
// (+ pad); weight gradient, one scale per column of the tile.
template <int kSbN>
struct alignas(16) ScaleSlot {   // 16-byte cp.async destinations, float2 reads
    float sa[kBM];   // scale of each row of the tile, this K block
    float sb[kSbN];
};

template <int kMode>
struct Smem {
    uint64_t full[kStages], empty[kStages];
    uint64_t sfull[kSSlots], sempty[kSSlots];
    uint64_t tfull[2], tempty[2], xchg[2], drain;
    uint32_t tmem_base;
    int abort;
    int total_items;
    float amax[2][4][128];
    ScaleSlot<kMode == kModeFP8W ? kBN : 4> scales[kSSlots];
    int prefix[kMaxGroups + 1];
    int offs[kMaxGroups + 1];   // row offsets of the groups (weight gradient: K-block offsets)
};
// The weight gradient's tiles have 2-3 K blocks and 128 KB of fp32 output each:
// a 2-stage ring, and 4 KB per epilogue warp to stage its output for TMA stores.
template <int kMode>
__host__ __device__ constexpr int stages_of() {
    return kMode == kModeFP8W ? 2 : kStages;
}
template <int kMode>
__host__ __device__ constexpr size_t ring_bytes() {
    return size_t(stages_of<kMode>()) * (kABytes + kBBytes);
}
constexpr size_t kStageBytes = 4096;   // one warp's 32 rows x 128 bytes, 128-byte swizzle
template <int kMode>
__host__ __device__ constexpr size_t staging_offset() {   // from the ring's start, 1024-byte aligned
    return (ring_bytes<kMode>() + sizeof(Smem<kMode>) + 1023) / 1024 * 1024;
}
template <int kMode>
__host__ __device__ constexpr size_t smem_bytes() {
    return staging_offset<kMode>() + (kMode == kModeFP8W ? kEpiWarps * kStageBytes : 0) + 1024;
}
static_assert(smem_bytes<kModeFP8W>() <= 227 * 1024 && smem_bytes<kModeFP8>() <= 227 * 1024, "shared memory");
static_assert(offsetof(Smem<kModeFP8W>, scales) % 16 == 0 && sizeof(ScaleSlot<kBN>) % 16 == 0, "scale slots");

struct Item {
    int g, mt, nt, sp;
};

// m_tiles_fixed > 0: every group has that many row tiles (weight gradient)
template <class S>
__device__ __forceinline__ Item decode(int item, const S& s, int G, int n_tiles_n, int splits, int m_tiles_fixed = 0) {
    int lo = 0, hi = G;  // prefix[lo] <= item < prefix[hi]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (s.prefix[mid] <= item) lo = mid;
        else hi = mid;
    }
    Item it;
    it.g = lo;
    int local = item - s.prefix[lo];
    it.sp = local % splits;
    local /= splits;
    if (m_tiles_fixed > 0) {
        // weight gradient: N tiles first, so that the CTAs running side by side write
        // whole rows of the fp32 output (its HBM stream) rather than scattered pieces
        it.nt = local % n_tiles_n;
        it.mt = local / n_tiles_n;
        return it;
    }
    // row tiles first: the CTAs running side by side share the weight tiles (L2)
    int m_tiles = (s.offs[lo + 1] - s.offs[lo] + kBM - 1) / kBM;
    it.mt = local % m_tiles;
    it.nt = local / m_tiles;
    return it;
}

// x * sigmoid(x) with CUDA's fast exp and divide intrinsics (about 2 ulp): the result
// feeds a 1x128 E4M3 quantisation (or a bf16 rounding), far coarser than that error.
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// 32 bytes to global memory in one instruction (address 32-byte aligned).
__device__ __forceinline__ void st_global_32B(void* p, const uint32_t* w) {   // w[0..7]
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

template <int kMode, int kEpi, bool kGather = false>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem<kMode>& s = *reinterpret_cast<Smem<kMode>*>(ring + ring_bytes<kMode>());
    constexpr bool kW = kMode == kModeFP8W;         // weight gradient: groups split K
    constexpr bool kScaled = kMode != kModeBF16;     // FP8 operands with scales
    constexpr int kSt = stages_of<kMode>();
    const uint32_t staging = smem_u32(ring + staging_offset<kMode>());
    const uint32_t ringA = smem_u32(ring);
    const uint32_t ringB = ringA + kSt * kABytes;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = args.G;
    const int n_tiles_n = args.Nd / kBN;
    const int splits = args.splits;
    const int steps_per_split = (args.k_steps + splits - 1) / splits;
    const int m_fixed = kW ? int(args.M_total / kBM) : 0;
    volatile int* abort = &s.abort;

    // ---------------- prologue ----------------
    if (threadIdx.x == 0) {
        // a gathered A arrives by cp.async: its stage gets a second arrival on full[]
        const uint32_t full_count = kGather ? 2u : 1u;
        for (int i = 0; i < kSt; ++i) {
            mbar_init(smem_u32(&s.full[i]), full_count);
            mbar_init(smem_u32(&s.empty[i]), 1);
        }
        for (int i = 0; i < kSSlots; ++i) {
            mbar_init(smem_u32(&s.sfull[i]), 32);         // one cp.async arrival per producer lane
            mbar_init(smem_u32(&s.sempty[i]), kEpiWarps * 32);   // every epilogue lane arrives
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s.tfull[i]), 1);
            mbar_init(smem_u32(&s.tempty[i]), kEpiWarps * 32);
            mbar_init(smem_u32(&s.xchg[i]), kEpiWarps * 32);
        }
        mbar_init(smem_u32(&s.drain), 1);
        s.abort = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&s.tmem_base), 512);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 0) {
        // group row offsets and the running count of work items per group
        int running = 0;
        bool bad = false;
        for (int base = 0; base <= G; base += 32) {
            int g = base + lane;
            int off = 0;
            if (g <= G) {
                off = args.group_offsets ? args.group_offsets[g] : (g == 0 ? 0 : (int)args.M_total);
                s.offs[g] = off;
            }
            __syncwarp();
            int items = 0;
            if (g < G) {
                int nxt = args.group_offsets ? args.group_offsets[g + 1] : (int)args.M_total;
                int rows = nxt - off;
                if (kW) {
                    // K-block offsets; every group owns all M/128 x Nd/256 output tiles
                    // (a group without tokens writes zeros)
                    if (rows < 0 || off < 0 || nxt > args.k_steps) bad = true;
                    items = m_fixed * n_tiles_n;
                } else {
                    if (rows < 0 || off < 0 || nxt > args.M_total) bad = true;
                    items = rows > 0 ? ((rows + kBM - 1) / kBM) * n_tiles_n * splits : 0;
                }
            }
            int incl = items;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (g <= G) s.prefix[g] = running + incl - items;
            running += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (args.group_offsets && args.group_offsets[0] != 0) bad = true;
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
            s.total_items = bad ? 0 : running;
            if (bad && blockIdx.x == 0) report(MOE_ERR_DEVICE_DATA);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s.tmem_base;
    const int total = s.total_items;

    if (kGather && warp == kProducerWarp) {
        // ---------------- A rows gathered by cp.async (every lane), B by TMA (lane 0) ----------------
        // Row m of a tile is row a_gather[r] (routed rows r) or r - a_gather_tk (the shared
        // expert's) of a_src; rows past the group's end read zeros (computed, never stored).
        // Lane l copies rows l, l+32, l+64, l+96, all eight 16-byte pieces of each, into the
        // layout the MMA descriptor reads: piece c of row m at c ^ (m % 8) (the 128-byte
        // swizzle TMA would write). A stage gets its second arrival once this lane's copies
        // into it have landed and a proxy fence has made them visible to the tensor core;
        // copies run kAhead stages ahead of those arrivals. Measured at the V3 shape this
        // feeds GEMM 1 at well under the TMA path's rate (4.8 against 2.8 ms): the one warp's
        // copies and their completion waits, not the MMA, set the pace. Variants that were
        // slower still: kAhead = 3 (the MMA then waits on every stage's arrival), and copies
        // of four whole rows per warp instruction through a shared row table.
        constexpr int kAhead = 2;
        int stage = 0, sig = 0, pending = 0;
        uint32_t phase = 0;
        int armed[kStages] = {0, 0, 0, 0};
        bool stop = false;
        auto signal_oldest = [&]() {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s.full[sig]));
            if (++sig == kSt) sig = 0;
            --pending;
        };
        for (int item = blockIdx.x; item < total && !stop; item += gridDim.x) {
            const Item it = decode(item, s, G, n_tiles_n, splits);
            const int a_row = s.offs[it.g] + it.mt * kBM;
            const int rows = s.offs[it.g + 1] - a_row;
            const int b_row = it.g * args.Nd + it.nt * kBN;
            const uint8_t* src[4];
            uint32_t nbytes[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = lane + 32 * i;
                src[i] = args.a_src;
                nbytes[i] = 0u;
                if (m < rows) {
                    const int64_t r = int64_t(a_row) + m;
                    const int64_t tok = r < args.a_gather_tk ? int64_t(__ldg(args.a_gather + r)) : r - args.a_gather_tk;
                    src[i] = args.a_src + tok * int64_t(args.Kd);
                    nbytes[i] = 16u;
                }
            }
            const int k0 = it.sp * steps_per_split;
            const int k1 = min(args.k_steps, k0 + steps_per_split);
            for (int ks = k0; ks < k1; ++ks) {
                int ok = 1;
                if (lane == 0) ok = mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, abort);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    stop = true;
                    break;
                }
                if (lane == 0) {
                    const uint32_t fb = smem_u32(&s.full[stage]);
                    mbar_arrive_expect_tx(fb, kBBytes);
                    tma_load_2d(ringB + stage * kBBytes, &tmB, fb, ks * args.elems_per_step, b_row);
                    armed[stage] += 1;
                }
                const uint32_t dst = ringA + stage * kABytes;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int m = lane + 32 * i;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        cp_async_16z(dst + uint32_t(m * 128 + ((c ^ (m & 7)) * 16)), src[i] + ks * 128 + c * 16,
                                     nbytes[i]);
                }
                cp_async_commit();
                if (++pending > kAhead) {
                    cp_async_wait_group<kAhead>();   // the oldest pending stage's copies have landed
                    signal_oldest();
                }
                if (++stage == kSt) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        cp_async_wait_all();   // no copy into shared memory may outlive the block
        while (pending > 0) signal_oldest();
        // never leave the block while a TMA copy into its shared memory is in flight
        if (lane == 0)
            for (int i = 0; i < kSt; ++i)
                if (armed[i] > 0) mbar_wait_limit(smem_u32(&s.full[i]), uint32_t(armed[i] - 1) & 1u, 200000000ull);
        __syncwarp();
    } else if (warp == kProducerWarp) {
        // ---------------- TMA producer: one lane, nothing else in its loop ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int armed[kStages] = {0, 0, 0, 0};   // the first kSt are used
            bool stop = false;
            for (int item = blockIdx.x; item < total && !stop; item += gridDim.x) {
                const Item it = decode(item, s, G, n_tiles_n, splits, m_fixed);
                const int a_row = kW ? it.mt * kBM : s.offs[it.g] + it.mt * kBM;
                const int b_row = kW ? it.nt * kBN : it.g * args.Nd + it.nt * kBN;
                // weight gradient: the group's own K blocks, at its K-block offset
                const int kbase = kW ? s.offs[it.g] : 0;
                const int k0 = kW ? 0 : it.sp * steps_per_split;
                const int k1 = kW ? s.offs[it.g + 1] - s.offs[it.g] : min(args.k_steps, k0 + steps_per_split);
                int ka = k0 / args.a_k_repeat;   // A's K step
                int rep = k0 - ka * args.a_k_repeat;
                for (int ks = k0; ks < k1; ++ks) {
                    if (!mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, abort)) {
                        stop = true;
                        break;
                    }
                    const uint32_t fb = smem_u32(&s.full[stage]);
                    mbar_arrive_expect_tx(fb, kABytes + kBBytes);
                    tma_load_2d(ringA + stage * kABytes, &tmA, fb, (kbase + ka) * args.elems_per_step, a_row);
                    tma_load_2d(ringB + stage * kBBytes, &tmB, fb, (kbase + ks) * args.elems_per_step, b_row);
                    armed[stage] += 1;
                    if (++rep == args.a_k_repeat) {
                        rep = 0;
                        ++ka;
                    }
                    if (++stage == kSt) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // never leave the block while a copy into its shared memory is in flight
            for (int i = 0; i < kSt; ++i)
                if (armed[i] > 0) mbar_wait_limit(smem_u32(&s.full[i]), uint32_t(armed[i] - 1) & 1u, 200000000ull);
        }
        __syncwarp();
    } else if (warp == kScaleWarp) {
        // ---------------- FP8 scales: each K block's 128 row scales and 2 weight scales ----------------
        // copied into the shared ring by all 32 lanes (cp.async), ahead of the epilogue
        if constexpr (kW) {
            // weight gradient: 128 row scales and 256 column scales per K block, 16-byte copies
            int sslot = 0;
            uint32_t sphase = 0;
            bool stop = false;
            for (int item = blockIdx.x; item < total && !stop; item += gridDim.x) {
                const Item it = decode(item, s, G, n_tiles_n, splits, m_fixed);
                const float* sa_src = args.sa + it.mt * kBM + 4 * lane;
                const float* sb_src = args.sb + it.nt * kBN + 8 * lane;
                const int kb0 = s.offs[it.g], kb1 = s.offs[it.g + 1];
                for (int kb = kb0; kb < kb1; ++kb) {
                    int ok = 1;
                    if (lane == 0) ok = mbar_wait(smem_u32(&s.sempty[sslot]), sphase ^ 1u, abort);
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        stop = true;
                        break;
                    }
                    cp_async_16(smem_u32(&s.scales[sslot].sa[4 * lane]), sa_src + int64_t(kb) * args.lda_s);
                    const float* sbk = sb_src + int64_t(kb) * args.Nd;
                    cp_async_16(smem_u32(&s.scales[sslot].sb[8 * lane]), sbk);
                    cp_async_16(smem_u32(&s.scales[sslot].sb[8 * lane + 4]), sbk + 4);
                    cp_async_arrive_noinc(smem_u32(&s.sfull[sslot]));
                    if (++sslot == kSSlots) {
                        sslot = 0;
                        sphase ^= 1u;
                    }
                }
            }
            cp_async_wait_all();   // no copy into shared memory may outlive the block
        } else if constexpr (kMode == kModeFP8) {
            int sslot = 0;
            uint32_t sphase = 0;
            const int nkb = args.Kd / 128;
            bool stop = false;
            for (int item = blockIdx.x; item < total && !stop; item += gridDim.x) {
                const Item it = decode(item, s, G, n_tiles_n, splits);
                const int a_row = s.offs[it.g] + it.mt * kBM;
                // rows past a group's end are clamped into the matrix: computed, never stored;
                // a gathered A takes its rows' scales from the same source rows
                const float* sa_src[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    int64_t r = min(int64_t(a_row) + 4 * lane + i, args.M_total - 1);
                    if (kGather)
                        r = r < args.a_gather_tk ? int64_t(__ldg(args.a_gather + r)) : r - args.a_gather_tk;
                    sa_src[i] = args.sa + r;
                }
                const float* sb_src = args.sb + (int64_t(it.g) * (args.Nd / 128) + 2 * it.nt) * nkb;
                // the same K blocks as the MMA warp and the epilogue: this split's own
                const int k0 = it.sp * steps_per_split;
                const int k1 = min(args.k_steps, k0 + steps_per_split);
                for (int ks = k0; ks < k1; ++ks) {
                    int ok = 1;
                    if (lane == 0) ok = mbar_wait(smem_u32(&s.sempty[sslot]), sphase ^ 1u, abort);
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        stop = true;
                        break;
                    }
                    const int64_t koff = int64_t(ks) * args.lda_s;
                    const uint32_t dst = smem_u32(&s.scales[sslot].sa[4 * lane]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) cp_async_4(dst + 4 * i, sa_src[i] + koff);
                    if (lane == 0) {
                        cp_async_4(smem_u32(&s.scales[sslot].sb[0]), sb_src + ks);
                        cp_async_4(smem_u32(&s.scales[sslot].sb[1]), sb_src + nkb + ks);
                    }
                    cp_async_arrive_noinc(smem_u32(&s.sfull[sslot]));
                    if (++sslot == kSSlots) {
                        sslot = 0;
                        sphase ^= 1u;
                    }
                }
            }
            cp_async_wait_all();   // no copy into shared memory may outlive the block
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---------------- tcgen05.mma issuer: lane 0 alone ----------------
        // Only lane 0 waits and issues, so a wait that gives up cannot split the warp.
        if (lane == 0) {
            constexpr uint32_t idesc = kScaled ? make_idesc(0, 0, kBM, kBN) : make_idesc(1, 1, kBM, kBN);
            const int P = kScaled ? 1 : args.promote_steps;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_iter = 0;
            for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
                Item it = decode(item, s, G, n_tiles_n, splits, m_fixed);
                const int k0 = kW ? 0 : it.sp * steps_per_split;
                const int k1 = kW ? s.offs[it.g + 1] - s.offs[it.g] : min(args.k_steps, k0 + steps_per_split);
                uint32_t buf = acc_iter & 1u;
                bool ok = true;
                for (int ks = k0; ks < k1; ++ks) {
                    // one TMEM partial per chunk of P K steps (FP8: every 128-K block)
                    const bool first = (ks - k0) % P == 0;
                    const bool last = (ks - k0) % P == P - 1 || ks == k1 - 1;
                    if (first) {
                        buf = acc_iter & 1u;
                        if (!mbar_wait(smem_u32(&s.tempty[buf]), ((acc_iter >> 1) & 1u) ^ 1u, abort)) {
                            ok = false;
                            break;
                        }
                    }
                    if (!mbar_wait(smem_u32(&s.full[stage]), phase, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = smem_desc_sw128(ringA + stage * kABytes);
                    const uint64_t bd = smem_desc_sw128(ringB + stage * kBBytes);
                    const uint32_t d = tmem_base + buf * kBN;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t acc = (k > 0 || !first) ? 1u : 0u;
                        if (kScaled) mma_e4m3(d, ad + 2 * k, bd + 2 * k, idesc, acc);
                        else mma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, acc);
                    }
                    tc_commit(smem_u32(&s.empty[stage]));
                    if (last) {
                        tc_commit(smem_u32(&s.tfull[buf]));
                        acc_iter += 1;
                    }
                    if (++stage == kSt) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            // every issued MMA must be complete before TMEM is freed
            tc_commit(smem_u32(&s.drain));
            mbar_wait_limit(smem_u32(&s.drain), 0, 200000000ull);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue warps ----------------
        const int q = warp & 3;        // TMEM lane quarter = rows 32q..32q+31
        const int wg = warp >> 2;      // column slice
        // SwiGLU tiles pair columns c and 128 + c (gate and up of one output), so a
        // warp takes 32wg..32wg+31 and 128+32wg..128+32wg+31; the other epilogues
        // give a warp the 64 contiguous columns 64wg..64wg+63.
        constexpr bool kContig = (kEpi == MOE_EPI_BF16 || kEpi == MOE_EPI_F32);
        const uint32_t slice = kContig ? wg * 64 : wg * 32;
        const int row_in_tile = q * 32 + lane;
        const uint32_t lane_addr = tmem_base + (uint32_t(q * 32) << 16);
        uint32_t acc_iter = 0, tile_iter = 0;
        int sslot = 0;
        uint32_t sphase = 0;
        for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
            int k0, k1;
            {
                const Item it = decode(item, s, G, n_tiles_n, splits, m_fixed);
                k0 = kW ? 0 : it.sp * steps_per_split;
                k1 = kW ? s.offs[it.g + 1] - s.offs[it.g] : min(args.k_steps, k0 + steps_per_split);
            }
            float acc[64];
            bool ok = true;
            if constexpr (kW) {
                // weight gradient: each 128-K block's partial sums times
                // sa[row, kb] * sb[col, kb] (one scale per column), added into fp32 registers
                float2 acc2[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) acc2[i] = make_float2(0.0f, 0.0f);
                for (int ks = k0; ks < k1; ++ks) {
                    bool got = mbar_wait(smem_u32(&s.sfull[sslot]), sphase, abort);
                    const uint32_t buf = acc_iter & 1u;
                    got = got && mbar_wait(smem_u32(&s.tfull[buf]), (acc_iter >> 1) & 1u, abort);
                    if (!__all_sync(0xffffffffu, got)) {   // warp-collective TMEM loads follow
                        ok = false;
                        break;
                    }
                    const float sa_v = s.scales[sslot].sa[row_in_tile];
                    const float2 sa2 = make_float2(sa_v, sa_v);
                    tc_fence_after();
                    const uint32_t col = lane_addr + buf * kBN + slice;
                    // 4 columns per TMEM load: the per-column scales leave no registers for
                    // wider loads (16 columns spilled, and ran 1.6x slower)
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        uint32_t r[4];
                        tmem_ld_4(col + c * 4, r);
                        tmem_wait_ld(r);
                        if (c == 15) {
                            tc_fence_before();
                            mbar_arrive(smem_u32(&s.tempty[buf]));
                        }
                        const float2* sbp = reinterpret_cast<const float2*>(&s.scales[sslot].sb[slice + 4 * c]);
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const float2 f2 = __fmul2_rn(sbp[i], sa2);
                            acc2[c * 2 + i] = __ffma2_rn(
                                make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), f2,
                                acc2[c * 2 + i]);
                        }
                    }
                    // the slot is released after the last column scale was read
                    mbar_arrive(smem_u32(&s.sempty[sslot]));
                    if (++sslot == kSSlots) {
                        sslot = 0;
                        sphase ^= 1u;
                    }
                    acc_iter += 1;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    acc[2 * i] = acc2[i].x;
                    acc[2 * i + 1] = acc2[i].y;
                }
            } else if constexpr (kMode == kModeFP8) {
                // promotion (accumulation paragraph): each 128-K block's partial sums,
                // times sa[row, kb] * sb[nblk, kb], added into fp32 registers
                float2 acc2[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) acc2[i] = make_float2(0.0f, 0.0f);
                for (int ks = k0; ks < k1; ++ks) {
                    bool got = mbar_wait(smem_u32(&s.sfull[sslot]), sphase, abort);
                    float fl = 0.0f, fh = 0.0f;
                    if (got) {
                        const float sa_v = s.scales[sslot].sa[row_in_tile];
                        fl = sa_v * s.scales[sslot].sb[0];
                        fh = sa_v * s.scales[sslot].sb[1];
                        // each lane releases the slot after its own reads (no warp barrier and
                        // no single-lane branch in the promotion loop)
                        mbar_arrive(smem_u32(&s.sempty[sslot]));
                    }
                    if (++sslot == kSSlots) {
                        sslot = 0;
                        sphase ^= 1u;
                    }
                    const uint32_t buf = acc_iter & 1u;
                    got = got && mbar_wait(smem_u32(&s.tfull[buf]), (acc_iter >> 1) & 1u, abort);
                    // the TMEM loads below are warp-collective: the warp goes on only if
                    // every lane saw both waits complete, and gives up as one otherwise
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t col = lane_addr + buf * kBN + slice;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        // paired slices: chunks 0,1 in the first weight block, 2,3 in the
                        // second; contiguous slices lie in block wg / 2
                        uint32_t r[16];
                        tmem_ld_16(col + (kContig ? c * 16 : (c >> 1) * 128 + (c & 1) * 16), r);
                        tmem_wait_ld(r);
                        if (c == 3) {
                            tc_fence_before();
                            mbar_arrive(smem_u32(&s.tempty[buf]));
                        }
                        const float f = kContig ? (wg < 2 ? fl : fh) : (c < 2 ? fl : fh);
                        const float2 f2 = make_float2(f, f);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            acc2[c * 8 + i] = __ffma2_rn(
                                make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), f2,
                                acc2[c * 8 + i]);
                    }
                    acc_iter += 1;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    acc[2 * i] = acc2[i].x;
                    acc[2 * i + 1] = acc2[i].y;
                }
            } else {
                // bf16: the partial sums of each chunk of P K steps are added into fp32
                // registers (fp32 accumulation in TMEM over at most P * 64 products)
                const int P = args.promote_steps;
                float2 acc2[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) acc2[i] = make_float2(0.0f, 0.0f);
                for (int c0 = k0; c0 < k1; c0 += P) {
                    const uint32_t buf = acc_iter & 1u;
                    const bool got = mbar_wait(smem_u32(&s.tfull[buf]), (acc_iter >> 1) & 1u, abort);
                    if (!__all_sync(0xffffffffu, got)) {   // warp-collective TMEM loads follow
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t col = lane_addr + buf * kBN + slice;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t r[16];
                        tmem_ld_16(col + (kContig ? c * 16 : (c >> 1) * 128 + (c & 1) * 16), r);
                        tmem_wait_ld(r);
                        if (c == 3) {
                            tc_fence_before();
                            mbar_arrive(smem_u32(&s.tempty[buf]));
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            acc2[c * 8 + i] = __fadd2_rn(
                                acc2[c * 8 + i], make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])));
                    }
                    acc_iter += 1;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    acc[2 * i] = acc2[i].x;
                    acc[2 * i + 1] = acc2[i].y;
                }
            }
            if (!ok) break;

            // ---- epilogue of the tile (tile coordinates decoded again: fewer live registers) ----
            const Item it = decode(item, s, G, n_tiles_n, splits, m_fixed);
            const int row_local = it.mt * kBM + row_in_tile;
            // weight gradient: group g's output is rows g*M .. g*M+M-1 of C, all of them written
            const bool valid = kW || row_local < s.offs[it.g + 1] - s.offs[it.g];
            const int64_t grow = kW ? int64_t(it.g) * args.M_total + row_local : int64_t(s.offs[it.g]) + row_local;
            constexpr int ep = kEpi;
            if constexpr (ep == MOE_EPI_SWIGLU_FP8 || ep == MOE_EPI_SWIGLU_BF16) {
                if (ep == MOE_EPI_SWIGLU_FP8 && args.h_out && valid) {
                    // the products themselves, rounded to bf16, at their columns of the
                    // [M_total, Nd] product (gate columns, then the up columns 128 further)
                    uint16_t* hrow = args.h_out + grow * args.Nd + int64_t(it.nt) * kBN + wg * 32;
#pragma unroll
                    for (int half = 0; half < 2; ++half)
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            uint32_t w[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                w[i] = pack_bf16x2(acc[32 * half + 16 * v + 2 * i], acc[32 * half + 16 * v + 2 * i + 1]);
                            st_global_32B(hrow + 128 * half + 16 * v, w);
                        }
                }
                float a[32];
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    a[i] = silu(acc[i]) * acc[32 + i];
                    amax = fmaxf(amax, fabsf(a[i]));
                }
                const int64_t ocol = int64_t(it.nt) * 128 + wg * 32;
                const int64_t ldo = args.Nd / 2;
                if constexpr (ep == MOE_EPI_SWIGLU_FP8) {
                    const uint32_t par = tile_iter & 1u;
                    s.amax[par][wg][row_in_tile] = amax;
                    mbar_arrive(smem_u32(&s.xchg[par]));
                    const bool got = mbar_wait(smem_u32(&s.xchg[par]), (tile_iter >> 1) & 1u, abort);
                    if (!__all_sync(0xffffffffu, got)) break;   // the warp leaves the tile loop as one
                    amax = fmaxf(fmaxf(s.amax[par][0][row_in_tile], s.amax[par][1][row_in_tile]),
                                 fmaxf(s.amax[par][2][row_in_tile], s.amax[par][3][row_in_tile]));
                    const float sc = tile_scale(amax);
                    if (valid) {
                        uint8_t* out = reinterpret_cast<uint8_t*>(args.C) + grow * ldo + ocol;
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint32_t p0 = pack_e4m3x2(__fdiv_rn(a[4 * i], sc), __fdiv_rn(a[4 * i + 1], sc));
                            const uint32_t p1 =
                                pack_e4m3x2(__fdiv_rn(a[4 * i + 2], sc), __fdiv_rn(a[4 * i + 3], sc));
                            w[i] = p0 | (p1 << 16);
                        }
                        st_global_32B(out, w);
                        if (wg == 0) args.c_scales[int64_t(it.nt) * args.M_total + grow] = sc;
                    }
                } else if (valid) {
                    uint16_t* out = reinterpret_cast<uint16_t*>(args.C) + grow * ldo + ocol;
#pragma unroll
                    for (int v = 0; v < 2; ++v) {
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(a[16 * v + 2 * i], a[16 * v + 2 * i + 1]);
                        st_global_32B(out + 16 * v, w);
                    }
                }
            } else if constexpr (ep == MOE_EPI_BF16) {
                // A thread holds 128 bytes of its row. Four lanes swap 32-byte pieces
                // (a 4x4 transpose by two xor-shuffle rounds) so that in store i the lanes
                // 4a..4a+3 write the whole 128 bytes of row 4a+i: 8 full lines per store.
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
                const bool b0 = lane & 1, b1 = lane & 2;
#pragma unroll
                for (int c = 0; c < 4; c += 2)
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const uint32_t v = __shfl_xor_sync(0xffffffffu, b0 ? w[8 * c + r] : w[8 * c + 8 + r], 1);
                        if (b0) w[8 * c + r] = v;
                        else w[8 * c + 8 + r] = v;
                    }
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const uint32_t v = __shfl_xor_sync(0xffffffffu, b1 ? w[8 * c + r] : w[8 * c + 16 + r], 2);
                        if (b1) w[8 * c + r] = v;
                        else w[8 * c + 16 + r] = v;
                    }
                const int rows = s.offs[it.g + 1] - s.offs[it.g];
                const int64_t c0 = int64_t(it.nt) * kBN + slice + 16 * (lane & 3);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int rl = it.mt * kBM + q * 32 + (lane & ~3) + i;
                    if (rl < rows)
                        st_global_32B(reinterpret_cast<uint16_t*>(args.C) + (int64_t(s.offs[it.g]) + rl) * args.Nd + c0,
                                      w + 8 * i);
                }
            } else if (kW) {
                // weight gradient, fp32 [G][M][Nd], by TMA stores: the warp's 32 rows x 32
                // columns at a time go to its 4 KB staging buffer (lane = row, 16-byte
                // chunk c at c ^ (row % 8): the 128-byte swizzle of the store's tensor map,
                // no bank conflicts), and lane 0 stores the box while the warp goes on
                const uint32_t buf = staging + uint32_t(warp) * uint32_t(kStageBytes);
                const int32_t y0 = int32_t(int64_t(it.g) * args.M_total + it.mt * kBM + q * 32);
                const int32_t x0 = int32_t(it.nt * kBN + slice);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (lane == 0) bulk_wait_read_all();   // the buffer's last store has read it
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float* v = acc + 32 * half + 4 * c;
                        const uint32_t dst = buf + uint32_t(lane) * 128u + uint32_t((c ^ (lane & 7)) * 16);
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "f"(v[0]), "f"(v[1]),
                                     "f"(v[2]), "f"(v[3])
                                     : "memory");
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, buf, x0 + 32 * half, y0);
                        bulk_commit();
                    }
                }
            } else if (valid) {
                // MOE_EPI_F32: split-K partial sums, [splits][M_total][Nd]
                const int64_t c0 = int64_t(it.nt) * kBN + slice;
                float* out = reinterpret_cast<float*>(args.C) + (int64_t(it.sp) * args.M_total + grow) * args.Nd + c0;
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(acc[8 * v + i]);
                    st_global_32B(out + 8 * v, w);
                }
            }
            tile_iter += 1;
        }
    }

    // ---------------- teardown ----------------
    if (kW && warp < kEpiWarps && lane == 0) bulk_wait_all();   // every TMA store of this warp written
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

// 2-D K-major tensor map: `rows` rows of `inner` elements (row stride
// `row_bytes`), box = 128 bytes of K x `box_rows` rows, 128-byte swizzle,
// out-of-range rows read as zero.
bool make_kmajor_map(CUtensorMap* tm, const void* base, bool bf16, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                     uint32_t box_rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {bf16 ? 64u : 128u, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(tm, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                     const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int kMode, int kEpi, bool kGather = false>
static cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c, const GemmArgs& args,
                          int grid, cudaStream_t stream) {
    static PerDeviceOnce once;
    constexpr size_t kSmemBytes = smem_bytes<kMode>();
    cudaError_t e = allow_smem(once, grouped_gemm_kernel<kMode, kEpi, kGather>, int(kSmemBytes));
    if (e != cudaSuccess) return e;
    grouped_gemm_kernel<kMode, kEpi, kGather><<<grid, kThreads, kSmemBytes, stream>>>(a, b, c, args);
    return cudaGetLastError();
}

cudaError_t run_grouped_gemm(int mode, const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& args, int grid,
                             cudaStream_t stream, const CUtensorMap* c) {
    const CUtensorMap& cm = c ? *c : a;   // only the weight gradient stores through a tensor map
    if (mode == kModeFP8W) {
        if (args.epilogue == MOE_EPI_F32 && c) return launch<kModeFP8W, MOE_EPI_F32>(a, b, cm, args, grid, stream);
        return cudaErrorInvalidValue;
    }
    if (mode == kModeFP8) {
        if (args.epilogue == MOE_EPI_SWIGLU_FP8)
            return args.a_gather ? launch<kModeFP8, MOE_EPI_SWIGLU_FP8, true>(a, b, cm, args, grid, stream)
                                 : launch<kModeFP8, MOE_EPI_SWIGLU_FP8>(a, b, cm, args, grid, stream);
        if (args.epilogue == MOE_EPI_BF16)
            return args.a_gather ? launch<kModeFP8, MOE_EPI_BF16, true>(a, b, cm, args, grid, stream)
                                 : launch<kModeFP8, MOE_EPI_BF16>(a, b, cm, args, grid, stream);
        return cudaErrorInvalidValue;
    }
    if (args.epilogue == MOE_EPI_SWIGLU_BF16) return launch<kModeBF16, MOE_EPI_SWIGLU_BF16>(a, b, cm, args, grid, stream);
    if (args.epilogue == MOE_EPI_BF16) return launch<kModeBF16, MOE_EPI_BF16>(a, b, cm, args, grid, stream);
    if (args.epilogue == MOE_EPI_F32) return launch<kModeBF16, MOE_EPI_F32>(a, b, cm, args, grid, stream);
    return cudaErrorInvalidValue;
}

// 2-D fp32 row-major store map: `rows` rows of `cols` floats, box 32 x 32,
// 128-byte swizzle (the weight gradient's staged output).
bool make_f32_store_map(CUtensorMap* tm, void* base, uint64_t cols, uint64_t rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int gemm_max_groups() { return kMaxGroups; }

}  // namespace moe
