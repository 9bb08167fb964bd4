// moe_permute_static: the permutation of moe_permute with its scratch memory
// inside the library instead of in a caller workspace.
//
// Some callers cannot allocate device memory for a workspace: code whose
// device memory is owned entirely by another allocator that it cannot ask for
// a buffer (an embedding runtime, a framework that reserved the whole GPU for
// its own pool), and code that must not allocate once it is running, because
// cudaMalloc can synchronise the device, take milliseconds, or fail under
// memory pressure. This entry point serves them: the per-chunk expert
// histograms that moe_permute keeps in its workspace live here in a
// fixed-size array in the library's device memory.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds its 4 MiB until the process exits. Host code cannot use the
// array's name as a device address (it is a host-side stand-in), so the
// first call on each device looks up the real address with
// cudaGetSymbolAddress while that device is current, and later calls on that
// device reuse it. The cached address belongs to the context it was looked up
// in: it is dropped when a launch fails, and a caller that resets the device
// (cudaDeviceReset) must not call this entry point again in that process.
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int64_t kStaticScratchInts = int64_t(1) << 20;   // 4 MiB of int32

__device__ __align__(256) int32_t g_permute_scratch[kStaticScratchInts];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_permute_scratch on the current device (looked up once
// per device), or nullptr with the CUDA error in *err.
void* static_scratch(cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_permute_scratch);
        if (*err != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

// Forgets the current device's cached address, so that the next call looks it
// up again (after a failed launch, the context may have been torn down).
void forget_static_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    g_scratch_addr[dev] = nullptr;
}

}  // namespace

}  // namespace moe

extern "C" moe_status moe_permute_static(const uint16_t* x, int64_t T, int d, const int32_t* topk_idx, int N, int K,
                                         int out_dtype, int with_shared, int32_t* offsets, int32_t* perm_token,
                                         int32_t* dest_row, void* x_perm, float* x_perm_scales,
                                         moe_stream_t stream) {
    // the same argument rules as moe_permute
    REQUIRE(T >= 0 && T * (K + 1) <= kMaxRows, "moe_permute_static: T=%lld out of range", (long long)T);
    REQUIRE(d > 0 && d % 128 == 0, "moe_permute_static: d=%d must be a multiple of 128", d);
    REQUIRE(N >= 1 && N <= 1024, "moe_permute_static: N=%d must be in [1, 1024]", N);
    REQUIRE(K >= 1 && K <= 16 && K <= N, "moe_permute_static: K=%d", K);
    REQUIRE(out_dtype == MOE_DTYPE_BF16 || out_dtype == MOE_DTYPE_E4M3, "moe_permute_static: out dtype %d",
            out_dtype);
    REQUIRE(offsets, "moe_permute_static: null offsets");
    if (T > 0) {
        REQUIRE(x && topk_idx && perm_token && dest_row && x_perm, "moe_permute_static: null pointer");
        REQUIRE(out_dtype != MOE_DTYPE_E4M3 || x_perm_scales, "moe_permute_static: E4M3 output needs scales");
        REQUIRE(al16(x) && al16(x_perm), "moe_permute_static: x and x_perm must be 16-byte aligned");
    }
    const size_t need = moe::permute_ws_bytes(T, N);
    if (need > size_t(moe::kStaticScratchInts) * sizeof(int32_t))
        return fail(MOE_ERR_WORKSPACE,
                    "moe_permute_static: T=%lld, N=%d need %zu bytes of scratch; the built-in scratch holds %lld "
                    "bytes (ceil(T/32)*N + N <= %lld int32); use moe_permute with a workspace",
                    (long long)T, N, need, (long long)(moe::kStaticScratchInts * 4),
                    (long long)moe::kStaticScratchInts);
    cudaError_t e = cudaSuccess;
    void* scratch = moe::static_scratch(&e);
    if (!scratch) return fail(MOE_ERR_CUDA, "moe_permute_static: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    e = moe::launch_permute(x, T, d, topk_idx, N, K, out_dtype, with_shared ? 1 : 0, offsets, perm_token, dest_row,
                            x_perm, x_perm_scales, scratch, stream);
    if (e != cudaSuccess) {
        moe::forget_static_scratch();
        return fail(MOE_ERR_CUDA, "moe_permute_static: launch: %s", cudaGetErrorString(e));
    }
    return MOE_OK;
}
