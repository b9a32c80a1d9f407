// fa_merge_kernel.cuh -- merge of partial attention states computed over disjoint key ranges.
//
// Each split s left, for every query row, the state of the online softmax over its keys:
// m_s (reference maximum of the scaled scores, log2 units), l_s (sum of weights relative to
// m_s) and o_s (unnormalised weighted sum of V rows). Two states over disjoint key sets merge as
//   m = max(m_1, m_2),  l = l_1 2^(m_1 - m) + l_2 2^(m_2 - m),  o = o_1 2^(m_1 - m) + o_2 2^(m_2 - m)
// ("11. Fusion, recompute, and flash attention", section 11.6, last paragraph, and exercise 3;
// here in base 2, and folded over all splits at once). The answer is O = o / l, and the row's
// log-sum-exp is (m + log2 l) ln 2.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "fa_bounds.cuh"
#include "sm103_ptx.cuh"

namespace fa {

// Where the split units' rows live: split unit t is unit split_begin + t, numbered
// bh * num_units + u, whose rows are u * 256 + r for r < split_rows = min(256, nq).
struct MergeMap {
    int split_begin, num_units, split_rows, nq;
    int bh;  // slices of O (B * H)
    // Nonzero: signal the stream's next programmatic-dependent launch as soon as every block has
    // passed its wait (else at completion).
    int trigger_dependents;
};

// One warp per R consecutive merged rows; lane i owns D/32 consecutive columns of each. The
// splits are merged in groups of G: every load of a group (all R rows) is issued before any is
// used; within a group the states are merged against the group maximum, then the group is merged
// into the running state. R = 1 (G = 4) is the general form; R = 2 (G = 2) halves the number of
// warps, for merges whose one-row grid would not fit one wave of resident blocks.
template <int D, bool BF16, int R, int G>
__global__ void __launch_bounds__(256) fa_merge_kernel(const float* __restrict__ o_part,
                                                       const float* __restrict__ ml_part,
                                                       void* __restrict__ o, float* __restrict__ lse,
                                                       int64_t rows, int num_splits, MergeMap map) {
    constexpr int E = D / 32;
    // Launched as a programmatic dependent of the attention kernel: wait until that grid has
    // completed and its partial states are visible (a no-op for an ordinary launch).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // The next launch (the next attention call) may then take SMs as this grid's blocks leave; it
    // waits for this grid to complete before it reads or writes global memory.
    if (map.trigger_dependents) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // 32-bit index arithmetic: rows, units and query rows all fit in int (checked on the host).
    const int row0 = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * R;
    const int lane = threadIdx.x & 31;
    if (row0 >= rows) return;
    const float2* ml = reinterpret_cast<const float2*>(ml_part);
    float m[R], l[R], acc[R][E];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[r][e] = 0.f;
    }
    for (int s0 = 0; s0 < num_splits; s0 += G) {
        const int g = min(G, num_splits - s0);
        float2 st[R][G];
        float v[R][G][E];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int u = 0; u < G; ++u) {
                if (u < g && row0 + r < rows) {
                    const int64_t prow = static_cast<int64_t>(s0 + u) * rows + row0 + r;
                    st[r][u] = ml[prow];
                    const float* src = o_part + prow * D + lane * E;
                    if constexpr (E == 4) {
                        const float4 x = *reinterpret_cast<const float4*>(src);
                        v[r][u][0] = x.x; v[r][u][1] = x.y; v[r][u][2] = x.z; v[r][u][3] = x.w;
                    } else {
                        const float2 x = *reinterpret_cast<const float2*>(src);
                        v[r][u][0] = x.x; v[r][u][1] = x.y;
                    }
                } else {
                    st[r][u] = make_float2(-INFINITY, 0.f);
#pragma unroll
                    for (int e = 0; e < E; ++e) v[r][u][e] = 0.f;
                }
            }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float m_new = m[r];
#pragma unroll
            for (int u = 0; u < G; ++u) m_new = fmaxf(m_new, st[r][u].x);
            const float c_old = (m[r] == -INFINITY) ? 0.f : ptx::ex2(m[r] - m_new);
            l[r] *= c_old;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[r][e] *= c_old;
#pragma unroll
            for (int u = 0; u < G; ++u) {
                const float w = (st[r][u].x == -INFINITY) ? 0.f : ptx::ex2(st[r][u].x - m_new);
                l[r] += st[r][u].y * w;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[r][e] += w * v[r][u][e];
            }
            m[r] = m_new;
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int row = row0 + r;
        if (row >= rows) break;
        const int tu = row / map.split_rows;
        const int unit = map.split_begin + tu;
        const int bh = unit / map.num_units;
        const int q_row = (unit - bh * map.num_units) * 256 + (row - tu * map.split_rows);
        if (q_row >= map.nq) continue;
        const int64_t out_row = static_cast<int64_t>(bh) * map.nq + q_row;
        if (!in_bounds(bh < map.bh, BOUNDS_MERGE_O, out_row)) continue;
        const float inv_l = (l[r] > 0.f) ? 1.f / l[r] : 0.f;
        uint32_t packed[E / 2];
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
            const float a = acc[r][2 * e] * inv_l, b = acc[r][2 * e + 1] * inv_l;
            if constexpr (BF16) {
                __nv_bfloat162 x = __floats2bfloat162_rn(a, b);
                packed[e] = *reinterpret_cast<uint32_t*>(&x);
            } else {
                __half2 x = __floats2half2_rn(a, b);
                packed[e] = *reinterpret_cast<uint32_t*>(&x);
            }
        }
        uint8_t* dst = static_cast<uint8_t*>(o) + (out_row * D + lane * E) * 2;
        if constexpr (E == 4) {
            *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
        } else {
            *reinterpret_cast<uint32_t*>(dst) = packed[0];
        }
        if (lse != nullptr && lane == 0) lse[out_row] = (m[r] + __log2f(l[r])) * 0.6931471805599453f;
    }
}

}  // namespace fa
