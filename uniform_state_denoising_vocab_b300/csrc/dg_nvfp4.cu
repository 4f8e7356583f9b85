// dg_nvfp4.cu -- NVFP4 operand preparation on the device:
//   quant_rows_nvfp4_kernel  two-level NVFP4 quantisation of bf16 rows (the E4M3 rule's 4-bit
//                            counterpart, applied to the hidden states in front of an NVFP4 head);
//   pack_scales_kernel       plain [rows][d/16] block scales -> the packed scale chunks the
//                            block-scaled MMA's tensor-memory copies consume;
//   repack_rowblock_kernel   packed scales of the slot rows -> the row-block layout the head
//                            reads for its A operand (the quantiser writes it directly when h
//                            is quantised inside a pass).
// The NVFP4 rule, in IEEE binary32: amax = max_k |h_k|; amax == 0 gives row scale 1 and all
// codes and block scales 0; otherwise g = fp32(amax / 2688) (2688 = 448 * 6) and, per block of
// 16 elements with bmax = max |h_k|, sb = e4m3_rn_satfinite(fp32(bmax / fp32(6 g))); a zero sb
// zeroes the block, else q_k = e2m1_rn_satfinite(fp32(h_k / fp32(value(sb) * g))). Element value
// = e2m1(q) * value(sb) * g. Codes are packed two per byte, element 2j in the low nibble.
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {
namespace {

constexpr int kQThreads = 128;

// Byte offset of (row, K block) in the packed layout: one 4096-byte chunk per (256-row group G,
// 256-element K slice s) at (G * d/256 + s) * 4096; inside it, with m = row % 256, l = m % 32,
// c = m / 32 and block = 16 s + 4 j + kb (j = 64-element MMA step of the slice):
//   (l / 8) * 1024 + j * 256 + (c / 4) * 128 + (l % 8) * 16 + (c % 4) * 4 + kb.
// Read as 8-row x 16-byte core matrices, a chunk holds for every step j the scale-factor tile of
// the 256 rows (lane l, column c) with 8-row groups 1024 bytes apart: the source of one 128x256b
// tensor-memory copy per step when four copies of the chunk sit 4096 bytes apart (one per lane
// quadrant), and of a 32x128b copy of one 128-row half from byte j * 256 + half * 128.
__device__ __forceinline__ size_t sf_offset(int row, int blk, int nslices) {
    const int G = row >> 8, m = row & 255, l = m & 31, c = m >> 5;
    const int s = blk >> 4, j = (blk >> 2) & 3, kb = blk & 3;
    return (static_cast<size_t>(G) * nslices + s) * 4096 + (l >> 3) * 1024 + j * 256 +
           (c >> 2) * 128 + (l & 7) * 16 + (c & 3) * 4 + kb;
}

// Byte offset of (row, K block) in the row-block layout of the head's A operand: per (128-row
// block b, 256-element K slice s, pair p of 64-element steps) a 4096-byte tile of 128 rows x 32
// bytes (8-row x 16-byte core matrices, 8-row groups 256 bytes apart, the second 16 bytes of a
// row 128 bytes on), read by one 128x256b tensor-memory copy into 8 columns. Row L = 32 q + l of
// the block holds the scales of step 2 p + jj at bytes jj * 16 + q * 4 .. + 3 of its 32: column
// 4 jj + q, the column the block-scaled MMA reads for lane quadrant q when the step's scale
// address is column 4 jj. The other bytes are never read.
//   ((b * d/256 + s) * 2 + p) * 4096 + (L / 8) * 256 + jj * 128 + (L % 8) * 16 + q * 4 + kb
__device__ __forceinline__ size_t sf_rowblock_offset(int row, int blk, int nslices) {
    const int b = row >> 7, L = row & 127;
    const int s = blk >> 4, j = (blk >> 2) & 3, kb = blk & 3;
    return ((static_cast<size_t>(b) * nslices + s) * 2 + (j >> 1)) * 4096 + (L >> 3) * 256 +
           (j & 1) * 128 + (L & 7) * 16 + (L >> 5) * 4 + kb;
}

__device__ __forceinline__ size_t sf_out_offset(int layout, int row, int blk, int nslices) {
    return layout == 0 ? sf_offset(row, blk, nslices) : sf_rowblock_offset(row, blk, nslices);
}

__device__ __forceinline__ float e4m3_value(uint8_t c) {
    __nv_fp8_e4m3 v;
    v.__x = c;
    return static_cast<float>(v);
}

__device__ __forceinline__ float block_max_q(float v, float* red) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    return fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
}

// Grid: one CTA of kQThreads per row of the scale layout (R rounded up to 256 for the packed
// layout, to 128 for the row-block layout); rows >= R only zero their block scales.
__global__ void __launch_bounds__(kQThreads)
    quant_rows_nvfp4_kernel(const __nv_bfloat16* __restrict__ h, int R, int d,
                            uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                            float* __restrict__ scale, uint32_t* status, int layout) {
    __shared__ float red[4];
    grid_dependency_wait();
    grid_launch_dependents();
    const int r = blockIdx.x;
    const int nb = d / 16, nsl = d / 256;
    if (r >= R) {
        for (int b = threadIdx.x; b < nb; b += kQThreads) sf[sf_out_offset(layout, r, b, nsl)] = 0;
        return;
    }
    const uint4* hr = reinterpret_cast<const uint4*>(h + static_cast<size_t>(r) * d);
    float amax = 0.f;
    bool bad = false;
    for (int c = threadIdx.x; c < d / 8; c += kQThreads) {
        const uint4 v = hr[c];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float a = __uint_as_float(w[i] << 16), b = __uint_as_float(w[i] & 0xFFFF0000u);
            bad |= !isfinite(a) || !isfinite(b);
            amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(b)));
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(status, DG_ST_NONFINITE);
    amax = block_max_q(amax, red);
    uint2* qr = reinterpret_cast<uint2*>(q + static_cast<size_t>(r) * (d / 2));
    if (amax == 0.f) {
        for (int b = threadIdx.x; b < nb; b += kQThreads) {
            qr[b] = make_uint2(0u, 0u);
            sf[sf_out_offset(layout, r, b, nsl)] = 0;
        }
        if (threadIdx.x == 0) scale[r] = 1.0f;
        return;
    }
    const float g = __fdiv_rn(amax, 2688.0f);
    const float g6 = __fmul_rn(6.0f, g);
    for (int b = threadIdx.x; b < nb; b += kQThreads) {
        const uint4 v0 = hr[2 * b], v1 = hr[2 * b + 1];
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float x[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
        float bmax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(x[i]));
        const uint8_t sb = static_cast<uint8_t>(
            __nv_cvt_float_to_fp8(__fdiv_rn(bmax, g6), __NV_SATFINITE, __NV_E4M3));
        sf[sf_out_offset(layout, r, b, nsl)] = sb;
        const float sv = e4m3_value(sb);
        uint32_t packed[2] = {0u, 0u};
        if (sv != 0.f) {
            const float db = __fmul_rn(sv, g);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t c = static_cast<uint32_t>(
                                       __nv_cvt_float_to_fp4(__fdiv_rn(x[i], db), __NV_E2M1,
                                                             cudaRoundNearest)) & 0xFu;
                packed[i >> 3] |= c << (4 * (i & 7));
            }
        }
        qr[b] = make_uint2(packed[0], packed[1]);
    }
    if (threadIdx.x == 0) scale[r] = g;
}

// One thread per (padded row, block): plain [rows][d/16] -> packed chunks; rows >= rows_in get 0.
__global__ void pack_scales_kernel(const uint8_t* __restrict__ plain, int rows_in, int rows_pad,
                                   int d, uint8_t* __restrict__ packed) {
    const int nb = d / 16, nsl = d / 256;
    const size_t total = static_cast<size_t>(rows_pad) * nb;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(i / nb), b = static_cast<int>(i % nb);
        packed[sf_offset(r, b, nsl)] = r < rows_in ? plain[i] : 0;
    }
}

// One thread per (row of the row-block layout, block): packed -> row-block; rows >= R get 0.
__global__ void repack_rowblock_kernel(const uint8_t* __restrict__ packed, int R, int rows_out,
                                       int d, uint8_t* __restrict__ out) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int nb = d / 16, nsl = d / 256;
    const size_t total = static_cast<size_t>(rows_out) * nb;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(i / nb), b = static_cast<int>(i % nb);
        out[sf_rowblock_offset(r, b, nsl)] = r < R ? packed[sf_offset(r, b, nsl)] : 0;
    }
}

}  // namespace

int nvfp4_rows_pad(int rows) { return (rows + 255) / 256 * 256; }

size_t nvfp4_rowblock_bytes(int rows, int d) {
    return static_cast<size_t>((rows + 127) / 128) * 128 * (d / 16) * 4;
}

cudaError_t launch_quant_rows_nvfp4(const uint16_t* h, int R, int d, uint8_t* q, uint8_t* sf,
                                    float* scale, uint32_t* status, cudaStream_t stream,
                                    int layout) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(layout == 0 ? nvfp4_rows_pad(R) : (R + 127) / 128 * 128);
    cfg.blockDim = dim3(kQThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    set_pdl_attr(&attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quant_rows_nvfp4_kernel,
                              reinterpret_cast<const __nv_bfloat16*>(h), R, d, q, sf, scale, status,
                              layout);
}

cudaError_t launch_repack_rowblock(const uint8_t* packed, int R, int d, uint8_t* out,
                                   cudaStream_t stream) {
    const int rows_out = (R + 127) / 128 * 128;
    const size_t total = static_cast<size_t>(rows_out) * (d / 16);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((total + 255) / 256 < 148 * 8 ? (total + 255) / 256
                                                                            : 148 * 8));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    set_pdl_attr(&attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, repack_rowblock_kernel, packed, R, rows_out, d, out);
}

cudaError_t launch_pack_scales(const uint8_t* plain, int rows, int d, uint8_t* packed,
                               cudaStream_t stream) {
    const int rows_pad = nvfp4_rows_pad(rows);
    const size_t total = static_cast<size_t>(rows_pad) * (d / 16);
    const int blocks = static_cast<int>((total + 255) / 256 < 148 * 16 ? (total + 255) / 256 : 148 * 16);
    pack_scales_kernel<<<blocks, 256, 0, stream>>>(plain, rows, rows_pad, d, packed);
    return cudaGetLastError();
}

}  // namespace dg
