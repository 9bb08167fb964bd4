// Host-side interface of the tcgen05 grouped GEMM kernel (gemm.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// kModeFP8W: FP8 weight gradient, groups split K (group_offsets in 128-K blocks),
// scales per (K block, row of A) and per (K block, row of B), fp32 output [G][M][Nd].
enum { kModeFP8 = 0, kModeBF16 = 1, kModeFP8W = 2 };

// bf16 GEMMs add their TMEM partial sums into fp32 registers every this many
// 64-wide K steps (512 products): a long fp32 accumulation in the tensor
// cores alone drifts by ~1e-5 relative over the 21,504-term routing gate.
constexpr int kBf16PromoteSteps = 8;

struct GemmArgs {
    const int32_t* group_offsets;  // [G+1] device; nullptr = one group of M_total rows
    int G;
    int64_t M_total;
    int Nd;              // output columns per group, multiple of 256
    int Kd;              // K extent of B in elements (FP8: also of A)
    int k_steps;         // 128-byte K steps per output tile (before split)
    int a_k_repeat;      // B steps per A step: A's step = step / a_k_repeat (1 for a plain GEMM;
                         // the routing gate's B interleaves its split terms per 64-column block)
    int elems_per_step;  // 128 (e4m3) or 64 (bf16)
    int splits;          // split-K parts (MOE_EPI_F32 only; else 1)
    int promote_steps;   // bf16: K steps accumulated in TMEM before adding into fp32 registers
    int epilogue;        // MOE_EPI_*
    const float* sa;     // FP8: [Kd/128][lda_s] activation scales
    int64_t lda_s;
    const float* sb;     // FP8: [G][Nd/128][Kd/128] weight scales; FP8W: [Kd/128][Nd]
    void* C;
    float* c_scales;     // MOE_EPI_SWIGLU_FP8: [Nd/256][M_total]
    uint16_t* h_out;     // MOE_EPI_SWIGLU_FP8, optional: the fp32 products rounded to bf16 [M_total][Nd]
    // FP8, optional: A's rows gathered from a_src [a_rows][Kd]: row r of the grouped A
    // is row a_gather[r] of it (r < a_gather_tk) or row r - a_gather_tk (the shared
    // expert's rows); sa then has one column per row of a_src (lda_s = a_rows).
    // nullptr: A is read through its tensor map as it stands.
    const int32_t* a_gather;
    int64_t a_gather_tk;
    const uint8_t* a_src;
};

bool make_kmajor_map(CUtensorMap* tm, const void* base, bool bf16, uint64_t inner, uint64_t rows,
                     uint64_t row_bytes, uint32_t box_rows);

// c: the output's store map (kModeFP8W only, make_f32_store_map); nullptr otherwise.
cudaError_t run_grouped_gemm(int mode, const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& args, int grid,
                             cudaStream_t stream, const CUtensorMap* c = nullptr);
bool make_f32_store_map(CUtensorMap* tm, void* base, uint64_t cols, uint64_t rows);

int gemm_max_groups();

}  // namespace moe
