// fa_rope_kernel.cuh -- rotary position embedding of 16-bit rows, the prologue of attention with
// rotary positions ("Attention", phobos stdlib docs, "Rotary position embeddings").
//
//   form 0, rotate-half (`rope`): a row is [a | b], halves of D/2; pair i is (a_i, b_i).
//   form 1, interleaved pairs (`rope_pairs`): pair i is (x_{2i}, x_{2i+1}).
//   x0' = x0 cos - x1 sin,  x1' = x1 cos + x0 sin,  with cos/sin of row n's pair i taken from
//   fp32 tables [N][D/2] (the same table for every batch and head).
// Both elements of a pair are read before either is written, so in-place use is safe. The
// arithmetic is fp32, rounded once to the 16-bit type. Memory-bound: each thread moves 8 pairs
// (32 bytes of X, 64 bytes of tables) with 16-byte accesses.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "fa_bounds.cuh"

namespace fa {

template <bool BF16>
__device__ __forceinline__ float2 to_f2(uint32_t u) {
    if constexpr (BF16) {
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
    } else {
        return __half22float2(*reinterpret_cast<const __half2*>(&u));
    }
}

template <bool BF16>
__device__ __forceinline__ uint32_t from_f2(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

// One pair rotated in fp32: (x0, x1) -> (x0 cos - x1 sin, x1 cos + x0 sin). Each second product
// is rounded and the first is fused with the sum (explicit intrinsics, so that every kernel that
// rotates -- this pass and the attention kernel's prologue on Q -- gives the same bits).
__device__ __forceinline__ float2 rope_rotate(float x0, float x1, float c, float s) {
    return make_float2(__fmaf_rn(x0, c, -__fmul_rn(x1, s)), __fmaf_rn(x1, c, __fmul_rn(x0, s)));
}

// Rotate-half: four 32-bit words of the first half (a) and of the second half (b) of a row,
// 8 pairs whose angles are cs[0..8), sn[0..8).
template <bool BF16>
__device__ __forceinline__ void rope_half8(const uint32_t (&a)[4], const uint32_t (&b)[4],
                                           const float* cs, const float* sn, uint32_t (&ao)[4],
                                           uint32_t (&bo)[4]) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float2 fa = to_f2<BF16>(a[w]), fb = to_f2<BF16>(b[w]);
        const float2 lo = rope_rotate(fa.x, fb.x, cs[2 * w], sn[2 * w]);
        const float2 hi = rope_rotate(fa.y, fb.y, cs[2 * w + 1], sn[2 * w + 1]);
        ao[w] = from_f2<BF16>(lo.x, hi.x);
        bo[w] = from_f2<BF16>(lo.y, hi.y);
    }
}

// Rotate-half, 4 pairs: two 32-bit words of the first half (a) and of the second half (b).
template <bool BF16>
__device__ __forceinline__ void rope_half4(const uint32_t (&a)[2], const uint32_t (&b)[2],
                                           const float* cs, const float* sn, uint32_t (&ao)[2],
                                           uint32_t (&bo)[2]) {
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        const float2 fa = to_f2<BF16>(a[w]), fb = to_f2<BF16>(b[w]);
        const float2 lo = rope_rotate(fa.x, fb.x, cs[2 * w], sn[2 * w]);
        const float2 hi = rope_rotate(fa.y, fb.y, cs[2 * w + 1], sn[2 * w + 1]);
        ao[w] = from_f2<BF16>(lo.x, hi.x);
        bo[w] = from_f2<BF16>(lo.y, hi.y);
    }
}

// Interleaved pairs: n 32-bit words, one pair each, angles cs[0..n), sn[0..n).
template <bool BF16, int N>
__device__ __forceinline__ void rope_pairs_n(const uint32_t (&x)[N], const float* cs,
                                             const float* sn, uint32_t (&y)[N]) {
#pragma unroll
    for (int w = 0; w < N; ++w) {
        const float2 f = to_f2<BF16>(x[w]);
        const float2 r = rope_rotate(f.x, f.y, cs[w], sn[w]);
        y[w] = from_f2<BF16>(r.x, r.y);
    }
}

// Grid-stride over (row, group of 8 pairs). x, y: [rows_total][d] (y may equal x);
// cos_t, sin_t: [n][d/2], row r uses table row r % n.
template <bool BF16, int FORM>
__global__ void __launch_bounds__(256) fa_rope_kernel(const uint16_t* x, uint16_t* y,
                                                      const float* __restrict__ cos_t,
                                                      const float* __restrict__ sin_t,
                                                      int64_t rows_total, int64_t n, int d) {
    // Launched as a programmatic dependent: X may come from the stream's previous kernel.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int half = d / 2;
    const int groups = half / 8;  // groups of 8 pairs per row (a power of two: d/16)
    const int shift = __ffs(groups) - 1;
    const int64_t total = rows_total * groups;
    // The grid-stride loop walks rows; the row within its slice advances by the same stride
    // modulo n, so no 64-bit division runs per element.
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    int64_t nrow = (g >> shift) % n;
    const int64_t nstep_rows = stride >> shift;  // stride is a multiple of groups
    const int64_t nstep = nstep_rows % n;
    for (; g < total; g += stride) {
        const int64_t row = g >> shift;
        const int i0 = static_cast<int>(g & (groups - 1)) * 8;  // first pair of the group
        const float* ct = cos_t + nrow * half + i0;
        const float* st = sin_t + nrow * half + i0;
        nrow += nstep;
        if (nrow >= n) nrow -= n;
        const float4 c0 = *reinterpret_cast<const float4*>(ct);
        const float4 c1 = *reinterpret_cast<const float4*>(ct + 4);
        const float4 s0 = *reinterpret_cast<const float4*>(st);
        const float4 s1 = *reinterpret_cast<const float4*>(st + 4);
        const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        const uint16_t* src = x + row * d;
        uint16_t* dst = y + row * d;
        if (!in_bounds(row < rows_total && nrow < n && i0 + 8 <= half, BOUNDS_ROPE, row)) continue;
        if constexpr (FORM == 0) {
            // 8 elements of each half: a_i0.. and b_i0..
            const uint4 a = *reinterpret_cast<const uint4*>(src + i0);
            const uint4 b = *reinterpret_cast<const uint4*>(src + half + i0);
            const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
            uint32_t ao[4], bo[4];
            rope_half8<BF16>(av, bv, cs, sn, ao, bo);
            *reinterpret_cast<uint4*>(dst + i0) = make_uint4(ao[0], ao[1], ao[2], ao[3]);
            *reinterpret_cast<uint4*>(dst + half + i0) = make_uint4(bo[0], bo[1], bo[2], bo[3]);
        } else {
            // 16 consecutive elements = pairs i0..i0+7, one pair per 32-bit word
            const uint4 p0 = *reinterpret_cast<const uint4*>(src + 2 * i0);
            const uint4 p1 = *reinterpret_cast<const uint4*>(src + 2 * i0 + 8);
            const uint32_t pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
            uint32_t po[8];
            rope_pairs_n<BF16, 8>(pv, cs, sn, po);
            *reinterpret_cast<uint4*>(dst + 2 * i0) = make_uint4(po[0], po[1], po[2], po[3]);
            *reinterpret_cast<uint4*>(dst + 2 * i0 + 8) = make_uint4(po[4], po[5], po[6], po[7]);
        }
    }
}

}  // namespace fa
