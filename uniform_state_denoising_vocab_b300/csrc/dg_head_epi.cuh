// dg_head_epi.cuh -- the epilogue step shared by the tensor-core head kernels: fold one
// accumulator tile (this thread's TMEM lane = one slot row, BN fp32 columns = BN vocabulary ids)
// into the row's running softmax state, 32 columns per tcgen05.ld.
#pragma once
#include "dg_common.cuh"
#include "dg_ptx.cuh"

namespace dg {

// Per-warp copy of the tile's E4M3 column scales (w_scale[n] for the BN ids of the tile).
// Warp-local (no cross-warp barrier), so an aborting warp can never strand the others; the
// previous tile's reads of `csc` finished before the first __syncwarp.
template <int BN>
__device__ __forceinline__ void stage_column_scales(float* csc, const float* w_scale, int n_base,
                                                    int V, int lane) {
    __syncwarp();
    for (int j = lane; j < BN; j += 32) {
        const int n = n_base + j;
        csc[j] = (n < V) ? w_scale[n] : 0.f;
    }
    __syncwarp();
}

// taddr0: TMEM address of column 0 of this tile in this warp's lane quadrant.
// valid_tile: vocabulary ids of the tile inside [0, V) (may exceed BN).
template <int KIND, int BN>
__device__ __forceinline__ void drain_tile(RowState& st, uint32_t taddr0, const float* csc,
                                           float crow, int n_base, int valid_tile) {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        __syncwarp();
        tmem_ld32(taddr0 + c * 32, v);
        if (KIND == 1) {
            const float2* c2 = reinterpret_cast<const float2*>(csc + c * 32);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float2 sc = c2[j];
                mul_x2(v[2 * j], v[2 * j + 1], v[2 * j], v[2 * j + 1], sc.x, sc.y);
            }
        }
        const int valid = valid_tile - c * 32;
        if (valid >= 32)
            row_state_update<false>(st, v, crow, n_base + c * 32, 32);
        else if (valid > 0)
            row_state_update<true>(st, v, crow, n_base + c * 32, valid);
    }
}

// The same fold for NCOL columns already loaded into registers (v, multiple of 32 columns), so
// that the accumulator can be handed back to the MMAs before the arithmetic runs.
template <int KIND, int NCOL>
__device__ __forceinline__ void fold_columns(RowState& st, float (&v)[NCOL], const float* csc,
                                             float crow, int n_base, int valid_tile) {
#pragma unroll
    for (int c = 0; c < NCOL / 32; ++c) {
        float(&w)[32] = *reinterpret_cast<float(*)[32]>(v + c * 32);
        if (KIND == 1) {
            const float2* c2 = reinterpret_cast<const float2*>(csc + c * 32);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float2 sc = c2[j];
                mul_x2(w[2 * j], w[2 * j + 1], w[2 * j], w[2 * j + 1], sc.x, sc.y);
            }
        }
        const int valid = valid_tile - c * 32;
        if (valid >= 32)
            row_state_update<false>(st, w, crow, n_base + c * 32, 32);
        else if (valid > 0)
            row_state_update<true>(st, w, crow, n_base + c * 32, valid);
    }
}

}  // namespace dg
