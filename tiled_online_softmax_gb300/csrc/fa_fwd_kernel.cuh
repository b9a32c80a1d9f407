// fa_fwd_kernel.cuh -- the sm_103a attention forward kernel (tiled online softmax).
//
// One CTA owns one tile of BM = 128 query rows of one (batch, head) slice and streams the
// slice's keys past it in tiles of BN = 128 ("11. Fusion, recompute, and flash attention",
// section 11.9: one thread block per block of query rows, the query block loaded once, key
// blocks looped over). Per key tile j:
//
//   S_j = Q K_j^T                       tcgen05 MMA, fp32 accumulator in tensor memory (TMEM)
//   m_new = max(m, rowmax S_j * c)      c = scale * log2(e); every exponential is then a bare
//   corr  = 2^(m - m_new)               exp2 (same chapter, section 11.7: base 2 with log2 e
//   P_j   = 2^(S_j * c - m_new)         folded into the scale)
//   l     = l * corr + rowsum P_j
//   O     = O * corr + P_j V_j          the rescale runs on O in TMEM, then a second MMA adds
//                                       P_j V_j with P_j read from TMEM
//
// and after the last tile O / l is written once ("Flash Attention 2", "Write the data back to
// HBM": the division happens once at write-back). The recurrence is the one of section 11.6
// "Online softmax" taken one key block at a time ("Flash Attention 2", "Overview of the
// algorithm"; phobos "Attention", `online_softmax`).
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t of the tile (TMEM lane t), so row max and
//              row sum need no shuffles; it also rescales its O row and writes the output.
//   warp 4     MMA issuer (one lane) and TMEM owner.
//   warp 5     TMA producer (one lane): Q once, then K and V tiles through a ring of stages.
//
// Tensor memory (512 columns x 128 lanes of 32 bit):
//   [0,128)    S buffer 0 (fp32); its first 64 columns take P (16-bit pairs) once S is read
//   [128,256)  S buffer 1, same
//   [256,256+D) O accumulator (fp32)
// Two S buffers let the MMA warp compute S_{j+1} while the softmax warps work on S_j.
//
// Masking: a key j >= Nk (partial last tile, phobos "Attention", `attention`) or, under causal
// masking, a key after the query (phobos "Causal attention") gets weight 0 and is left out of
// the row maximum; key tiles entirely after the tile's last query are never loaded.
//
// Every wait is bounded: past the time limit the waiting thread records a site code in the
// device error word, raises the CTA's abort flag, and every role winds down (waiting, bounded
// again, for its own in-flight copies and MMAs) before TMEM is freed and the CTA exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int BM = 128;               // query rows per tile = TMEM lanes
constexpr int BN = 128;               // keys per tile
constexpr int NUM_THREADS = 192;
constexpr int SOFTMAX_THREADS = 128;  // warps 0-3
constexpr int MMA_WARP = 4;
constexpr int LOAD_WARP = 5;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_S0 = 0, TMEM_S1 = 128, TMEM_O = 256;

// Wait-site codes written to the device error word (first timeout wins).
enum WaitSite : int {
    SITE_LOAD_K_EMPTY = 1,
    SITE_LOAD_V_EMPTY = 2,
    SITE_MMA_Q_FULL = 3,
    SITE_MMA_K_FULL = 4,
    SITE_MMA_P_FULL = 5,
    SITE_MMA_V_FULL = 6,
    SITE_SOFTMAX_S_FULL = 7,
    SITE_SOFTMAX_O_READY = 8,
    SITE_DRAIN = 9,
};

struct Params {
    void* o;                   // output [bh][nq][D]
    int* err;                  // device error word (site code of the first timeout)
    int bh;                    // B * H
    int nq, nk;
    int num_q_tiles;
    float scale_log2;          // scale * log2(e)
    unsigned long long timeout_ns;
};

template <int D, int STAGES>
struct Smem {
    static constexpr int COL_BLOCKS = D / 64;            // 128-byte (64-element) column blocks
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2;          // one K or V tile
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + Q_BYTES;
    static constexpr int V_OFF = K_OFF + STAGES * KV_BYTES;
    static constexpr int BAR_OFF = V_OFF + STAGES * KV_BYTES;
    // barrier indices
    static constexpr int B_Q_FULL = 0;
    static constexpr int B_K_FULL = 1;
    static constexpr int B_K_EMPTY = B_K_FULL + STAGES;
    static constexpr int B_V_FULL = B_K_EMPTY + STAGES;
    static constexpr int B_V_EMPTY = B_V_FULL + STAGES;
    static constexpr int B_S_FULL = B_V_EMPTY + STAGES;  // 2
    static constexpr int B_P_FULL = B_S_FULL + 2;        // 2
    static constexpr int B_O_READY = B_P_FULL + 2;
    static constexpr int B_DRAIN = B_O_READY + 1;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int TMEM_SLOT_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int ABORT_OFF = TMEM_SLOT_OFF + 4;
    static constexpr int BYTES = ABORT_OFF + 4;
    // +1024 slack for 1024-byte alignment; at least 116 KB so that two CTAs never share an SM
    // (each holds all 512 TMEM columns; a second one would stall in tcgen05.alloc).
    static constexpr int ALLOC_BYTES = (BYTES + 1024 > 116 * 1024) ? BYTES + 1024 : 116 * 1024;
};

// ---------------------------------------------------------------------------------------------
// bounded wait
// ---------------------------------------------------------------------------------------------
struct Ctl {
    volatile int* abort;   // CTA-wide abort flag in shared memory
    int* err;
    unsigned long long timeout_ns;
};

// Wait for phase `parity` of `bar`. Returns false on timeout (after recording `site`) or, when
// `honor_abort` is set, as soon as another thread of the CTA has aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& ctl, int site,
                                         bool honor_abort = true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (honor_abort && *ctl.abort) return false;
            if (ptx::globaltimer_ns() - t0 > ctl.timeout_ns) {
                *ctl.abort = 1;
                atomicCAS(ctl.err, 0, site);
                return false;
            }
        }
    }
}

// Warp-uniform variant: every lane waits; the warp proceeds only if all lanes succeeded.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const Ctl& ctl,
                                              int site) {
    const bool ok = wait_bar(bar, parity, ctl, site);
    return __all_sync(0xffffffffu, ok);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t u) {
    if constexpr (BF16) {
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
    } else {
        return __half22float2(*reinterpret_cast<const __half2*>(&u));
    }
}

// ---------------------------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------------------------
template <int D, bool BF16, bool CAUSAL, int STAGES>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const Params p) {
    using L = Smem<D, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = ptx::smem_u32(smem);
    auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * static_cast<uint32_t>(i); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::ABORT_OFF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::TMEM_SLOT_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Tile schedule. Causal: the longest rows first, spread over all slices; otherwise the tiles
    // of one slice are adjacent so its K/V stay hot in L2.
    int bh, qt;
    if constexpr (CAUSAL) {
        bh = blockIdx.x % p.bh;
        qt = p.num_q_tiles - 1 - static_cast<int>(blockIdx.x / p.bh);
    } else {
        qt = blockIdx.x % p.num_q_tiles;
        bh = blockIdx.x / p.num_q_tiles;
    }
    const int q0 = qt * BM;
    int n_tiles = (p.nk + BN - 1) / BN;
    if constexpr (CAUSAL) n_tiles = min(n_tiles, (q0 + BM - 1) / BN + 1);

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        ptx::mbar_init(bar(L::B_Q_FULL), 1);
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar(L::B_K_FULL + s), 1);
            ptx::mbar_init(bar(L::B_K_EMPTY + s), 1);
            ptx::mbar_init(bar(L::B_V_FULL + s), 1);
            ptx::mbar_init(bar(L::B_V_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(L::B_S_FULL + b), 1);
            ptx::mbar_init(bar(L::B_P_FULL + b), SOFTMAX_THREADS);
        }
        ptx::mbar_init(bar(L::B_O_READY), 1);
        ptx::mbar_init(bar(L::B_DRAIN), 1);
        ptx::fence_barrier_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == LOAD_WARP && lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
    }
    if (warp == MMA_WARP) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Ctl ctl{abort_flag, p.err, p.timeout_ns};

    if (warp == LOAD_WARP) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t sq = sbase + L::Q_OFF, sk = sbase + L::K_OFF, sv = sbase + L::V_OFF;
            ptx::mbar_arrive_expect_tx(bar(L::B_Q_FULL), L::Q_BYTES);
            for (int c = 0; c < L::COL_BLOCKS; ++c)
                ptx::tma_load_3d(sq + c * (BM * 128), &tm_q, c * 64, q0, bh, bar(L::B_Q_FULL));
            int issued = 0;
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % STAGES;
                const uint32_t ph = (j / STAGES) & 1;
                if (!wait_bar(bar(L::B_K_EMPTY + st), ph ^ 1, ctl, SITE_LOAD_K_EMPTY)) break;
                ptx::mbar_arrive_expect_tx(bar(L::B_K_FULL + st), L::KV_BYTES);
                for (int c = 0; c < L::COL_BLOCKS; ++c)
                    ptx::tma_load_3d(sk + st * L::KV_BYTES + c * (BN * 128), &tm_k, c * 64,
                                     j * BN, bh, bar(L::B_K_FULL + st));
                if (!wait_bar(bar(L::B_V_EMPTY + st), ph ^ 1, ctl, SITE_LOAD_V_EMPTY)) {
                    issued = 2 * j + 1;
                    break;
                }
                ptx::mbar_arrive_expect_tx(bar(L::B_V_FULL + st), L::KV_BYTES);
                for (int c = 0; c < L::COL_BLOCKS; ++c)
                    ptx::tma_load_3d(sv + st * L::KV_BYTES + c * (BN * 128), &tm_v, c * 64,
                                     j * BN, bh, bar(L::B_V_FULL + st));
                issued = 2 * j + 2;
            }
            if (*abort_flag) {
                // Drain: every copy this thread started must land before the CTA's shared
                // memory can be released. The last copy into each stage is the newest phase.
                wait_bar(bar(L::B_Q_FULL), 0, ctl, SITE_DRAIN, false);
                for (int t = (issued > 2 * STAGES ? issued - 2 * STAGES : 0); t < issued; ++t) {
                    const int j = t / 2, st = j % STAGES;
                    const uint32_t ph = (j / STAGES) & 1;
                    const int b = (t & 1) ? L::B_V_FULL + st : L::B_K_FULL + st;
                    wait_bar(bar(b), ph, ctl, SITE_DRAIN, false);
                }
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = ptx::idesc_f16(BF16, BM, BN, false, false);
            constexpr uint32_t IDESC_O = ptx::idesc_f16(BF16, BM, D, false, true);
            const uint32_t sq = sbase + L::Q_OFF, sk = sbase + L::K_OFF, sv = sbase + L::V_OFF;
            bool ok = wait_bar(bar(L::B_Q_FULL), 0, ctl, SITE_MMA_Q_FULL);

            // S_j = Q K_j^T: K = D in steps of 16 elements (32 bytes inside a 128-byte swizzle
            // row); Q and K tiles are K-major, 8-row swizzle atoms 1024 bytes apart.
            auto issue_s = [&](int j) {
                const int st = j % STAGES;
                const uint32_t d_tmem = tmem + ((j & 1) ? TMEM_S1 : TMEM_S0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * (BM * 128) + (kk % 4) * 32;
                    const uint64_t a = ptx::sdesc_sw128(sq + off, 16, 1024);
                    const uint64_t b = ptx::sdesc_sw128(
                        sk + st * L::KV_BYTES + (kk / 4) * (BN * 128) + (kk % 4) * 32, 16, 1024);
                    ptx::mma_ss(d_tmem, a, b, IDESC_S, kk > 0 ? 1u : 0u);
                }
            };
            // O += P_j V_j: K = BN keys in steps of 16; P_j is A, read from TMEM (16 keys = 8
            // columns of 16-bit pairs); V_j is B in MN-major (D contiguous) layout: 16 keys =
            // 16 rows of 128 bytes, the next 64 columns of D one column block (BN rows) away.
            auto issue_pv = [&](int j) {
                const int st = j % STAGES;
                const uint32_t p_tmem = tmem + ((j & 1) ? TMEM_S1 : TMEM_S0);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t b = ptx::sdesc_sw128(sv + st * L::KV_BYTES + kk * (16 * 128),
                                                        BN * 128, 1024);
                    ptx::mma_ts(tmem + TMEM_O, p_tmem + kk * 8, b, IDESC_O,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
            };

            if (ok) ok = wait_bar(bar(L::B_K_FULL + 0), 0, ctl, SITE_MMA_K_FULL);
            if (ok) {
                ptx::tc_fence_after();
                issue_s(0);
                ptx::mma_commit(bar(L::B_S_FULL + 0));
                ptx::mma_commit(bar(L::B_K_EMPTY + 0));
            }
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j + 1 < n_tiles) {
                    const int st1 = (j + 1) % STAGES;
                    ok = wait_bar(bar(L::B_K_FULL + st1), ((j + 1) / STAGES) & 1, ctl,
                                  SITE_MMA_K_FULL);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    issue_s(j + 1);
                    ptx::mma_commit(bar(L::B_S_FULL + ((j + 1) & 1)));
                    ptx::mma_commit(bar(L::B_K_EMPTY + st1));
                }
                ok = wait_bar(bar(L::B_P_FULL + (j & 1)), (j >> 1) & 1, ctl, SITE_MMA_P_FULL);
                if (!ok) break;
                const int st = j % STAGES;
                ok = wait_bar(bar(L::B_V_FULL + st), (j / STAGES) & 1, ctl, SITE_MMA_V_FULL);
                if (!ok) break;
                ptx::tc_fence_after();
                issue_pv(j);
                ptx::mma_commit(bar(L::B_O_READY));
                ptx::mma_commit(bar(L::B_V_EMPTY + st));
            }
            if (*abort_flag) {
                // Drain: wait until every MMA this thread issued has finished with TMEM/smem.
                ptx::mma_commit(bar(L::B_DRAIN));
                wait_bar(bar(L::B_DRAIN), 0, ctl, SITE_DRAIN, false);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ softmax warps
        const int t = threadIdx.x;  // row within the tile = TMEM lane
        const int row = q0 + t;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const float c = p.scale_log2;
        float m = -INFINITY;  // running max of the scaled scores (log2 units)
        float l = 0.f;        // running denominator
        bool ok = true;

        for (int j = 0; j < n_tiles; ++j) {
            const int b = j & 1;
            const uint32_t s_cols = tmem + lane_base + (b ? TMEM_S1 : TMEM_S0);
            ok = wait_bar_warp(bar(L::B_S_FULL + b), (j >> 1) & 1, ctl, SITE_SOFTMAX_S_FULL);
            if (!ok) break;
            ptx::tc_fence_after();

            uint32_t sr[4][32];
#pragma unroll
            for (int q = 0; q < 4; ++q) ptx::tmem_ld32(s_cols + q * 32, sr[q]);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 4; ++q) ptx::reg_fence(sr[q]);

            const int k0 = j * BN;
            // Keys of this tile that the row may see: [k0, k_end).
            int k_end = min(k0 + BN, p.nk);
            if constexpr (CAUSAL) k_end = min(k_end, row + 1);
            const int n_vis = k_end - k0;  // may be <= 0 only for padding rows past Nq
            const bool full_tile = (n_vis >= BN);

            // Tile maximum of the scaled scores over visible keys. Scaling by c >= 0 is monotone
            // in floating point, so the maximum is taken on the raw scores and scaled once
            // (for c < 0 the minimum plays that role).
            const bool neg = c < 0.f;
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float sv = neg ? -__uint_as_float(sr[q][i]) : __uint_as_float(sr[q][i]);
                    if (full_tile || q * 32 + i < n_vis) mx[i & 7] = fmaxf(mx[i & 7], sv);
                }
            float m_tile = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            m_tile = (m_tile == -INFINITY) ? -INFINITY : (neg ? -m_tile : m_tile) * c;
            const float m_new = fmaxf(m, m_tile);
            // An empty state (m = -inf) has nothing to rescale; an all-hidden row keeps m = -inf
            // and is given weight 0 below.
            const float corr = (m == -INFINITY) ? 0.f : ptx::ex2(m - m_new);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;

            float sum[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) sum[i] = 0.f;
            uint32_t pk[2][32];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float p0 = ptx::ex2(fmaf(__uint_as_float(sr[q][i]), c, -m_use));
                    float p1 = ptx::ex2(fmaf(__uint_as_float(sr[q][i + 1]), c, -m_use));
                    if (!full_tile) {
                        if (q * 32 + i >= n_vis) p0 = 0.f;
                        if (q * 32 + i + 1 >= n_vis) p1 = 0.f;
                    }
                    // l sums the same 16-bit-rounded weights the PV product uses, so the
                    // final O / l is an exact weighted average of V under those weights.
                    const uint32_t u = pack2<BF16>(p0, p1);
                    const float2 r = unpack2<BF16>(u);
                    sum[i & 7] += r.x;
                    sum[(i + 1) & 7] += r.y;
                    pk[q >> 1][(q & 1) * 16 + i / 2] = u;
                }
            }
            const float rowsum = ((sum[0] + sum[1]) + (sum[2] + sum[3])) +
                                 ((sum[4] + sum[5]) + (sum[6] + sum[7]));
            l = l * corr + rowsum;
            // P_j over the first 64 columns of this S buffer (all of S_j is already in registers).
            ptx::tmem_st32(s_cols + 0, pk[0]);
            ptx::tmem_st32(s_cols + 32, pk[1]);

            if (j > 0) {
                // O holds sum_{i<j} P_i V_i relative to the old max once PV_{j-1} is done.
                ok = wait_bar_warp(bar(L::B_O_READY), (j - 1) & 1, ctl, SITE_SOFTMAX_O_READY);
                if (!ok) break;
                ptx::tc_fence_after();
                if (__any_sync(0xffffffffu, corr != 1.f)) {
                    const uint32_t o_cols = tmem + lane_base + TMEM_O;
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) {
                        uint32_t orr[32];
                        ptx::tmem_ld32(o_cols + q * 32, orr);
                        ptx::tmem_wait_ld();
                        ptx::reg_fence(orr);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            orr[i] = __float_as_uint(__uint_as_float(orr[i]) * corr);
                        ptx::tmem_st32(o_cols + q * 32, orr);
                    }
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(L::B_P_FULL + b));
            m = m_new;
        }

        // ---------------------------------------------------------------- epilogue: O / l
        if (ok && n_tiles > 0) {
            ok = wait_bar_warp(bar(L::B_O_READY), (n_tiles - 1) & 1, ctl, SITE_SOFTMAX_O_READY);
        }
        if (ok && n_tiles > 0) {
            ptx::tc_fence_after();
            const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
            const uint32_t o_cols = tmem + lane_base + TMEM_O;
            uint8_t* out_row = static_cast<uint8_t*>(p.o) +
                               (static_cast<size_t>(bh) * p.nq + row) * (D * 2);
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t orr[32];
                ptx::tmem_ld32(o_cols + q * 32, orr);
                ptx::tmem_wait_ld();
                ptx::reg_fence(orr);
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    packed[i] = pack2<BF16>(__uint_as_float(orr[2 * i]) * inv_l,
                                            __uint_as_float(orr[2 * i + 1]) * inv_l);
                if (row < p.nq) {
                    uint4* dst = reinterpret_cast<uint4*>(out_row + q * 64);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                            packed[4 * v + 3]);
                }
            }
        }
        ptx::tmem_wait_st();  // no TMEM store of this warp may be pending at dealloc
    }

    // ---------------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace fa
