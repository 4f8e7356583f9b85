// dg_common.cuh -- device-side building blocks shared by the head kernels and the sampler
// kernels: the softmax-partial monoid, the online update over a chunk of logits, the
// SplitMix64 counter hash, and status bits.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/dgcanvas.h"

namespace dg {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x on the special-function unit (relative error about 2^-22; flushes subnormal results).
__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two fp32 lanes per instruction (the packed f32x2 arithmetic of the sm_100 family): each lane is
// rounded exactly as the scalar instruction rounds it, so a fold written with these gives the
// same bits as the scalar fold, in about half the instructions.
__device__ __forceinline__ void fma_x2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                       float c0, float c1) {
    asm("{\n\t.reg .b64 a, b, c, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add_x2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "add.rn.f32x2 d, a, b;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void mul_x2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Softmax statistics of one slot row over a subset of the vocabulary, in base-2 units:
// with x_n = l_n * log2(e) (logit l_n), mx = max_n x_n, idx = smallest n attaining the max,
//   s = sum_n 2^(x_n - mx),   u = sum_n 2^(x_n - mx) * (x_n - mx).
// Over the full vocabulary: conf = max_n p_n = 1/s and H = -sum p ln p = ln2 * (log2 s - u/s).
// Stored as 16 bytes {mx, s, u, idx}.
struct Partial {
    float mx, s, u;
    int32_t idx;
};

__device__ __forceinline__ float4 pack(const Partial& p) {
    return make_float4(p.mx, p.s, p.u, __int_as_float(p.idx));
}
__device__ __forceinline__ Partial unpack(const float4& f) {
    return Partial{f.x, f.y, f.z, __float_as_int(f.w)};
}

__device__ __forceinline__ Partial partial_empty() {
    return Partial{-INFINITY, 0.f, 0.f, 0x7FFFFFFF};
}

// Monoid merge: a (x) b. Associative up to rounding; equal maxima keep the lower index, so the
// merged argmax is the lowest vocabulary index attaining the maximum. The side with the larger
// maximum ("hi") keeps its terms as they are (its rescale factor is exactly 1); only the other
// side is rescaled, by 2^(lo.mx - hi.mx) <= 1 on the special-function unit.
__device__ __forceinline__ Partial partial_merge(const Partial& a, const Partial& b) {
    if (b.s == 0.f) return a;
    if (a.s == 0.f) return b;
    const bool a_hi = (a.mx > b.mx) || (a.mx == b.mx && a.idx <= b.idx);
    const Partial& hi = a_hi ? a : b;
    const Partial& lo = a_hi ? b : a;
    const float d = lo.mx - hi.mx;  // <= 0
    const float e = ex2_fast(d);
    Partial r;
    r.mx = hi.mx;
    r.idx = hi.idx;
    r.s = fmaf(lo.s, e, hi.s);
    r.u = fmaf(e, fmaf(lo.s, d, lo.u), hi.u);
    return r;
}

// Running per-row state kept in registers by a head kernel's epilogue thread. Values are first
// compared in the "w" domain (raw accumulator times column scale), which is monotone in the
// logit because the row factor crow = inv_temp * row_scale * log2(e) is positive.
struct RowState {
    float mw;   // max of w seen so far
    float mx;   // mw * crow (base-2 logit of the running max)
    float s, u;
    int32_t idx;
};

__device__ __forceinline__ RowState row_state_init() {
    return RowState{-INFINITY, -INFINITY, 0.f, 0.f, 0x7FFFFFFF};
}

// Fold 32 consecutive columns (vocabulary ids n0 .. n0+31) into the running state.
// Columns j >= valid are ignored (vocabulary tail). Chunks arrive in increasing n0 order, so a
// chunk maximum equal to the running maximum keeps the earlier (lower) index.
template <bool kMasked>
__device__ __forceinline__ void row_state_update(RowState& st, const float (&w)[32], float crow,
                                                 int32_t n0, int valid) {
    float cm = -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (!kMasked || j < valid) cm = fmaxf(cm, w[j]);
    if (cm > st.mw) {
        int j0 = 31;
#pragma unroll
        for (int j = 31; j >= 0; --j)
            if ((!kMasked || j < valid) && w[j] == cm) j0 = j;
        const float nmx = cm * crow;
        if (st.s > 0.f) {
            const float d = st.mx - nmx;  // <= 0
            const float a = exp2f(d);
            st.u = a * fmaf(st.s, d, st.u);
            st.s *= a;
        }
        st.mw = cm;
        st.mx = nmx;
        st.idx = n0 + j0;
    }
    const float nmx = -st.mx;
    // four running sums per quantity (column j goes to sum j % 4), two lanes per instruction
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        float t0, t1, t2, t3;
        fma_x2(t0, t1, w[j + 0], w[j + 1], crow, crow, nmx, nmx);
        fma_x2(t2, t3, w[j + 2], w[j + 3], crow, crow, nmx, nmx);
        float e0 = ex2_fast(t0), e1 = ex2_fast(t1), e2 = ex2_fast(t2), e3 = ex2_fast(t3);
        if (kMasked) {
            if (j + 0 >= valid) e0 = 0.f, t0 = 0.f;
            if (j + 1 >= valid) e1 = 0.f, t1 = 0.f;
            if (j + 2 >= valid) e2 = 0.f, t2 = 0.f;
            if (j + 3 >= valid) e3 = 0.f, t3 = 0.f;
        }
        add_x2(s0, s1, s0, s1, e0, e1);
        add_x2(s2, s3, s2, s3, e2, e3);
        fma_x2(u0, u1, e0, e1, t0, t1, u0, u1);
        fma_x2(u2, u3, e2, e3, t2, t3, u2, u3);
    }
    st.s += (s0 + s1) + (s2 + s3);
    st.u += (u0 + u1) + (u2 + u3);
}

__device__ __forceinline__ Partial row_state_partial(const RowState& st) {
    return Partial{st.mx, st.s, st.u, st.idx};
}

// ---------------------------------------------------------------------------------------------
// SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): one output from state x.
// ---------------------------------------------------------------------------------------------
__host__ __device__ __forceinline__ uint64_t sm64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Counter key of canvas row `row` at pass `pass`; the re-randomised token is key mod V.
__host__ __device__ __forceinline__ uint64_t draw_key(uint64_t seed, uint32_t pass, uint64_t row) {
    return sm64(sm64(sm64(seed) ^ static_cast<uint64_t>(pass)) ^ row);
}

constexpr uint32_t kInitPass = 0xFFFFFFFFu;

// Exact x mod V for a 64-bit x and 1 <= V < 2^31, without the 64-bit integer division routine.
// With x = hi * 2^32 + lo: t = (hi mod V) * 2^32 + lo has the same residue and t < V * 2^32, so
// the quotient q = floor(t / V) < 2^32. q is estimated in double precision with inv_v = RN(1/V)
// (relative error below 2^-50, so the estimate is within one of q) and the remainder corrected.
__device__ __forceinline__ uint32_t mod_u64_by_u32(uint64_t x, uint32_t V, double inv_v) {
    const uint32_t hi = static_cast<uint32_t>(x >> 32), lo = static_cast<uint32_t>(x);
    const uint64_t t = (static_cast<uint64_t>(hi % V) << 32) | lo;
    const uint64_t q = __double2ull_rz(__dmul_rn(__ull2double_rn(t), inv_v));
    int64_t r = static_cast<int64_t>(t) - static_cast<int64_t>(q * V);
    if (r < 0) r += V;
    if (r >= static_cast<int64_t>(V)) r -= V;
    return static_cast<uint32_t>(r);
}

__device__ __forceinline__ void flag_status(uint32_t* status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

}  // namespace dg
