// fa_bwd_kernel.cuh -- attention backward by recompute on sm_103a.
//
// The forward pass keeps no P; the backward recomputes it tile by tile from Q, K and the saved
// log-sum-exp ("11. Fusion, recompute, and flash attention", section 11.9, "Backward", and the
// exercise "Backward with recompute"). With P = exp(scale * Q K^T - LSE) row by row:
//   dV = P^T dO,   dP = dO V^T,   dS = P * (dP - D)  with D_i = sum_d dO_i O_i,
//   dQ = scale * dS K,   dK = scale * dS^T Q.
// Three kernels, no atomics (results are deterministic):
//   fa_bwd_prep_kernel  D_i and LSE_i * log2(e) per query row (padded rows: +inf and 0, so
//                       padded queries get P = 0 with no further mask).
//   fa_bwd_dkdv_kernel  one CTA per 128 keys: S^T = K Q_i^T and dP^T = V dO_i^T into TMEM,
//                       P^T and dS^T rounded to 16 bits over them, dV += P^T dO_i and
//                       dK += dS^T Q_i accumulating in TMEM, over every query block i.
//   fa_bwd_dq_kernel    one CTA per 128 queries: S = Q K_j^T (two TMEM buffers, computed ahead)
//                       and dP = dO V_j^T, dS over S, dQ += dS K_j, over every key block j.
// Warp roles (192 threads): warps 0-3 compute (thread r owns TMEM lane r: a key row in the
// first kernel, a query row in the second), warp 4 issues MMAs (an elected lane, predicated
// issue) and owns TMEM, warp 5 issues TMA copies. Every wait is bounded as in the forward kernel.
// The three kernels are launched back to back as programmatic dependents: the dK/dV kernel
// waits for the preprocessing before reading anything; the dQ kernel reads nothing the dK/dV
// kernel writes and does not wait for it, except in its last CTA, so that the dQ grid
// completes after the dK/dV grid.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

struct BwdParams {
    void* dq;             // [bh][nq][D]
    void* dk;             // [bh][nk][D]
    void* dv;             // [bh][nk][D]
    const float* lse2;    // [bh][nq_pad]: LSE * log2(e); +inf on rows >= nq
    const float* delta;   // [bh][nq_pad]: sum_d dO * O; 0 on rows >= nq
    int* err;
    int bh, nq, nk, nq_pad;
    float scale;          // softmax scale
    float scale_log2;     // scale * log2(e)
    unsigned long long timeout_ns;
    // After issuing its last loads, each CTA prefetches into L2 the resident and first streamed
    // blocks of CTA blockIdx.x + next_prefetch_stride, one wave later (0: none).
    int next_prefetch_stride;
    // The load lane initialises the barriers itself and issues the resident and first streamed
    // blocks before the CTA-wide barrier (0: after it).
    int early_loads;
};

constexpr int BWD_THREADS = 192;
constexpr int BWD_MMA_WARP = 4;
constexpr int BWD_LOAD_WARP = 5;
constexpr uint32_t BWD_TMEM_S = 0, BWD_TMEM_DP = 128, BWD_TMEM_A = 256, BWD_TMEM_B = 384;

enum BwdSite : int {
    SITE_BWD_LOAD = 21,
    SITE_BWD_MMA = 22,
    SITE_BWD_COMPUTE = 23,
    SITE_BWD_DRAIN = 24,
    SITE_BWD_SMEM_LAYOUT = 25,  // dynamic shared memory too little aligned for the layout: no work done
};

// ---------------------------------------------------------------------------------------------
// D_i and LSE2_i: D / 8 threads per (padded) query row, 16-byte loads of O and dO
// ---------------------------------------------------------------------------------------------
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const void* __restrict__ o,
                                                          const void* __restrict__ dout,
                                                          const float* __restrict__ lse,
                                                          float* __restrict__ lse2,
                                                          float* __restrict__ delta, int bh,
                                                          int nq, int nq_pad) {
    // Launched as a programmatic dependent: O and dO may come from the stream's previous kernel.
    // The dK/dV kernel, launched after this one the same way, may take SMs as soon as every block
    // here has started; it waits for this grid to complete before reading anything.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int TPR = D / 8;  // threads per row, 8 elements each
    const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / TPR;
    const int sub = threadIdx.x % TPR;
    const bool live = w < static_cast<int64_t>(bh) * nq_pad;
    const int64_t h = live ? w / nq_pad : 0, r = live ? w % nq_pad : 0;
    float acc = 0.f;
    if (live && r < nq) {
        const int64_t src = (h * nq + r) * D + sub * 8;
        const uint4 a = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(o) + src);
        const uint4 b = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(dout) + src);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = unpack2<BF16>(av[e]), y = unpack2<BF16>(bv[e]);
            acc = fmaf(x.x, y.x, acc);
            acc = fmaf(x.y, y.y, acc);
        }
    }
    // Sum over the TPR threads of the row (aligned groups within the warp).
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (live && sub == 0 && in_bounds(h < bh && r < nq_pad, BOUNDS_BWD_PREP, w)) {
        if (r < nq) {
            delta[w] = acc;
            lse2[w] = lse[h * nq + r] * 1.4426950408889634f;
        } else {
            lse2[w] = INFINITY;
            delta[w] = 0.f;
        }
    }
}

// Packed fp32 arithmetic of the compute warps (pairs of columns in one instruction).
// {d0, d1} = {a0, a1} * {b0, b1} + {c0, c1}, one packed fused multiply-add.
__device__ __forceinline__ void ffma2v(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                       float c0, float c1) {
    asm("{\n\t.reg .b64 a, b, c, d;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %5};\n\t"
        "mov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
// {d0, d1} = {p0, p1} * ({x0, x1} - {y0, y1}): a packed subtract, then a packed multiply.
__device__ __forceinline__ void fmulsub2(float& d0, float& d1, float p0, float p1, float x0, float x1,
                                         float y0, float y1) {
    asm("{\n\t.reg .b64 p, x, y, d;\n\t"
        "mov.b64 p, {%2, %3};\n\t"
        "mov.b64 x, {%4, %5};\n\t"
        "mov.b64 y, {%6, %7};\n\t"
        "sub.rn.f32x2 d, x, y;\n\t"
        "mul.rn.f32x2 d, p, d;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(p0), "f"(p1), "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}

// ---------------------------------------------------------------------------------------------
// shared memory of the two main kernels
// ---------------------------------------------------------------------------------------------
template <int D, bool CAUSAL>
struct BwdSmem {
    static constexpr int COL_BLOCKS = D / 64;
    static constexpr int TILE = 128 * D * 2;          // one 128-row tile of Q, K, V or dO
    // Q_i is read by S^T(i) and dK(i), dO_i by dP^T(i) and dV(i), which comes first; so Q gets
    // the deeper ring (three stages: Q_{i+3} loads while block i+1 runs) and dO two. Each Q stage
    // also holds the block's lse2 (128 floats, read for P^T), each dO stage its delta (read for
    // dS^T, after dP^T(i) has read dO_i): the compute warps never wait on a load themselves.
    // A dO stage is freed when dV(i) has run and the compute warps have read its delta.
    static constexpr int Q_STAGES = 3;
    static constexpr int DO_STAGES = 2;
    static constexpr int VEC_BYTES = 128 * 4;
    static constexpr int R0_OFF = 0;                   // K block (resident)
    static constexpr int R1_OFF = TILE;                // V block (resident)
    static constexpr int A_OFF = 2 * TILE;             // Q ring
    static constexpr int B_OFF = A_OFF + Q_STAGES * TILE;   // dO ring
    static constexpr int LSE_OFF = B_OFF + DO_STAGES * TILE;           // lse2 per Q stage
    static constexpr int DELTA_OFF = LSE_OFF + Q_STAGES * VEC_BYTES;  // delta per dO stage
    static constexpr int BAR_OFF = DELTA_OFF + DO_STAGES * VEC_BYTES;
    static constexpr int B_RES_FULL = 0;                       // resident tiles landed
    static constexpr int B_Q_FULL = 1;                         // [Q_STAGES]
    static constexpr int B_Q_EMPTY = B_Q_FULL + Q_STAGES;      // [Q_STAGES] dK(i) done
    static constexpr int B_DO_FULL = B_Q_EMPTY + Q_STAGES;     // [DO_STAGES] dO_i + delta
    static constexpr int B_DO_EMPTY = B_DO_FULL + DO_STAGES;   // [DO_STAGES] dV(i) + 4 warps
    static constexpr int B_S_FULL = B_DO_EMPTY + DO_STAGES;
    static constexpr int B_DP_FULL = B_S_FULL + 1;
    static constexpr int B_P_HALF = B_DP_FULL + 1;      // P^T of queries 0-63 stored
    static constexpr int B_P_FULL = B_P_HALF + 1;
    static constexpr int B_DS_FULL = B_P_FULL + 1;
    static constexpr int B_MMA_DONE = B_DS_FULL + 1;
    static constexpr int B_DRAIN = B_MMA_DONE + 1;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int TMEM_SLOT_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int ABORT_OFF = TMEM_SLOT_OFF + 4;
    static constexpr int BYTES = ABORT_OFF + 4;
    // Up to 1024 bytes of slack for aligning the base to 1024 bytes (the 128-byte swizzle atom
    // repeats every 8 rows), as far as the 227 KB limit allows; the kernel checks at run time
    // that the slack it needs is there.
    // At least 116 KB, so that two CTAs never share an SM: each holds all 512 TMEM columns.
    static constexpr int MAX_BYTES = 232448;
    static constexpr int FIT_BYTES = BYTES + 1024 <= MAX_BYTES ? BYTES + 1024 : MAX_BYTES;
    static constexpr int ALLOC_BYTES = FIT_BYTES > 116 * 1024 ? FIT_BYTES : 116 * 1024;
    static_assert(BYTES + 256 <= MAX_BYTES, "shared memory budget");
};

// Operand descriptors of a 128-row tile staged by TMA in 64-column blocks (128-byte swizzle).
// K-major use (the tile's D is the MMA's K): step kk of 16 elements.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
    return ptx::sdesc_sw128(tile + (kk / 4) * (128 * 128) + (kk % 4) * 32, 16, 1024);
}
// MN-major use (the tile's rows are the MMA's K, its D the N): step kk of 16 rows.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {
    return ptx::sdesc_sw128(tile + kk * (16 * 128), 128 * 128, 1024);
}

template <int D>
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap* map, int row, int slice,
                                         uint32_t bar) {
#pragma unroll
    for (int c = 0; c < D / 64; ++c) ptx::tma_load_3d(dst + c * (128 * 128), map, c * 64, row, slice, bar);
}

// Convert 32 fp32 registers to 16 words of 16-bit pairs.
template <bool BF16>
__device__ __forceinline__ void pack16(const float* f, uint32_t (&u)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) u[i] = pack2<BF16>(f[2 * i], f[2 * i + 1]);
}

// Write a 16-bit row of D values from TMEM columns (fp32) times `mul` to global memory.
template <int D, bool BF16>
__device__ __forceinline__ void store_row(uint32_t tmem_cols, float mul, void* dst_row, bool keep) {
#pragma unroll 1
    for (int q = 0; q < D / 16; ++q) {
        uint32_t o[16];
        ptx::tmem_ld16(tmem_cols + q * 16, o);
        ptx::tmem_wait_ld();
        ptx::reg_fence(o);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * mul, __uint_as_float(o[2 * i + 1]) * mul);
        if (keep) {
            uint4* d = reinterpret_cast<uint4*>(static_cast<uint8_t*>(dst_row) + q * 32);
            d[0] = make_uint4(w[0], w[1], w[2], w[3]);
            d[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
    }
}

template <int D>
__device__ __forceinline__ void zero_row(void* dst_row) {
    uint4* d = static_cast<uint4*>(dst_row);
#pragma unroll
    for (int i = 0; i < D / 8; ++i) d[i] = make_uint4(0, 0, 0, 0);
}

// Prologue of the dK/dV kernel: barriers, TMEM. Returns the TMEM base.
template <int D, bool CAUSAL, typename Prologue>
__device__ __forceinline__ uint32_t bwd_setup(uint8_t* smem, uint32_t sbase, uint32_t tmem_slot_addr,
                                              uint32_t* tmem_slot, volatile int* abort_flag,
                                              bool early, Prologue&& prologue) {
    using L = BwdSmem<D, CAUSAL>;
    auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * static_cast<uint32_t>(i); };
    const int warp = threadIdx.x >> 5;
    const int init_thread = early ? BWD_LOAD_WARP * 32 : 0;
    if (threadIdx.x == init_thread) {
        *abort_flag = 0;
        ptx::mbar_init(bar(L::B_RES_FULL), 1);
        for (int s = 0; s < L::Q_STAGES; ++s) {
            ptx::mbar_init(bar(L::B_Q_FULL + s), 1);
            ptx::mbar_init(bar(L::B_Q_EMPTY + s), 1);
        }
        for (int s = 0; s < L::DO_STAGES; ++s) {
            ptx::mbar_init(bar(L::B_DO_FULL + s), 1);
            ptx::mbar_init(bar(L::B_DO_EMPTY + s), 1 + 4);  // the dV commit and the 4 compute warps
        }
        ptx::mbar_init(bar(L::B_S_FULL), 1);
        ptx::mbar_init(bar(L::B_DP_FULL), 1);
        ptx::mbar_init(bar(L::B_P_HALF), 128);
        ptx::mbar_init(bar(L::B_P_FULL), 128);
        ptx::mbar_init(bar(L::B_DS_FULL), 128);
        ptx::mbar_init(bar(L::B_MMA_DONE), 1);
        ptx::mbar_init(bar(L::B_DRAIN), 1);
        ptx::fence_barrier_init();
        ptx::fence_proxy_async_smem();
    }
    // Early mode: the load lane, which initialised the barriers just above, starts its loads now.
    if (early && threadIdx.x == init_thread) prologue();
    if (warp == BWD_MMA_WARP) {
        ptx::tmem_alloc(tmem_slot_addr, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    return *tmem_slot;
}

__device__ __forceinline__ uint32_t elect_leader() {
    uint32_t leader;
    asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
                 : "=r"(leader));
    return leader;
}

// ---------------------------------------------------------------------------------------------
// dK, dV: one CTA per (slice, 128 keys); resident K (R0) and V (R1); ring A = Q_i, ring B = dO_i
// ---------------------------------------------------------------------------------------------
template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdParams p) {
    using L = BwdSmem<D, CAUSAL>;
    constexpr int QS = L::Q_STAGES, DS = L::DO_STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    if (pad + L::BYTES > static_cast<uint32_t>(L::ALLOC_BYTES)) {
        // Not enough slack to align the layout (never seen: the dynamic window starts 1024-byte
        // aligned). Report it and do nothing; no barrier or TMEM is in use yet.
        if (threadIdx.x == 0) atomicCAS(p.err, 0, SITE_BWD_SMEM_LAYOUT);
        return;
    }
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = ptx::smem_u32(smem);
    auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * static_cast<uint32_t>(i); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::ABORT_OFF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::TMEM_SLOT_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int nkb = (p.nk + 127) / 128, nqb = (p.nq + 127) / 128;
    // The CTAs of one slice are adjacent (they share Q and dO in L2). Under causal masking the
    // longest ones (kb = 0) come first within each slice; ordering them longest-first across all
    // slices instead measured 5 % slower on a 16 x 16384 launch (Q and dO of every slice in flight).
    const int bh = blockIdx.x / nkb, kb = blockIdx.x % nkb;
    const int k0 = kb * 128;
    const int i_begin = CAUSAL ? kb : 0;  // query blocks before the diagonal see none of these keys
    const int n = nqb > i_begin ? nqb - i_begin : 0;
    const bool early = p.early_loads != 0;
    // Loads of the load lane: the resident K and V blocks; query block `it` of Q (with its lse2
    // row) and of dO (with its delta row) into their stages.
    auto load_res = [&]() {
        ptx::mbar_arrive_expect_tx(bar(L::B_RES_FULL), 2 * L::TILE);
        tma_tile<D>(sbase + L::R0_OFF, &tm_k, k0, bh, bar(L::B_RES_FULL));
        tma_tile<D>(sbase + L::R1_OFF, &tm_v, k0, bh, bar(L::B_RES_FULL));
    };
    auto load_q_blk = [&](int it) {
        const int qs = it % QS;
        const size_t vo = static_cast<size_t>(bh) * p.nq_pad + static_cast<size_t>(i_begin + it) * 128;
        ptx::mbar_arrive_expect_tx(bar(L::B_Q_FULL + qs), L::TILE + L::VEC_BYTES);
        tma_tile<D>(sbase + L::A_OFF + qs * L::TILE, &tm_q, (i_begin + it) * 128, bh, bar(L::B_Q_FULL + qs));
        ptx::bulk_load(sbase + L::LSE_OFF + qs * L::VEC_BYTES, p.lse2 + vo, L::VEC_BYTES,
                       bar(L::B_Q_FULL + qs));
    };
    auto load_do_blk = [&](int it) {
        const int ds = it % DS;
        const size_t vo = static_cast<size_t>(bh) * p.nq_pad + static_cast<size_t>(i_begin + it) * 128;
        ptx::mbar_arrive_expect_tx(bar(L::B_DO_FULL + ds), L::TILE + L::VEC_BYTES);
        tma_tile<D>(sbase + L::B_OFF + ds * L::TILE, &tm_do, (i_begin + it) * 128, bh, bar(L::B_DO_FULL + ds));
        ptx::bulk_load(sbase + L::DELTA_OFF + ds * L::VEC_BYTES, p.delta + vo, L::VEC_BYTES,
                       bar(L::B_DO_FULL + ds));
    };
    bool pre = false;  // the resident blocks and query block 0 were issued before the barrier
    const uint32_t tmem = bwd_setup<D, CAUSAL>(smem, sbase, ptx::smem_u32(tmem_slot), tmem_slot,
                                               abort_flag, early, [&]() {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (n > 0) {
            load_res();
            load_q_blk(0);
            load_do_blk(0);
            pre = true;
        }
    });
    const Ctl ctl{abort_flag, p.err, p.timeout_ns};
    // Launched as a programmatic dependent of the preprocessing: its outputs (and Q, K, V, dO,
    // possibly from earlier kernels) are read only after it has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // The dQ kernel is launched as a programmatic dependent of this one and reads nothing this
    // kernel writes, so it may take SMs as soon as every CTA here has started (and, being past
    // the wait above, the preprocessing has completed).
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == BWD_LOAD_WARP) {
        if (lane == 0 && n > 0) {
            if (!pre) load_res();
            int issued_q = pre ? 1 : 0, issued_do = pre ? 1 : 0;
            for (int it = pre ? 1 : 0; it < n; ++it) {
                const int qs = it % QS, ds = it % DS;
                if (!wait_bar(bar(L::B_Q_EMPTY + qs), ((it / QS) & 1) ^ 1, ctl, SITE_BWD_LOAD)) break;
                load_q_blk(it);
                issued_q = it + 1;
                if (!wait_bar(bar(L::B_DO_EMPTY + ds), ((it / DS) & 1) ^ 1, ctl, SITE_BWD_LOAD)) break;
                load_do_blk(it);
                issued_do = it + 1;
            }
            // The CTA one wave later starts as this wave's CTAs leave: its K and V blocks and its
            // first Q and dO blocks, prefetched into L2 now that this CTA's loads are issued.
            const int nb = static_cast<int>(blockIdx.x) + p.next_prefetch_stride;
            if (p.next_prefetch_stride > 0 && nb < static_cast<int>(gridDim.x) && !*abort_flag) {
                const int nbh = nb / nkb, nk0 = (nb % nkb) * 128, nq0 = CAUSAL ? nk0 : 0;
                for (int c = 0; c < D / 64; ++c) {
                    ptx::tma_prefetch_3d(&tm_k, c * 64, nk0, nbh);
                    ptx::tma_prefetch_3d(&tm_v, c * 64, nk0, nbh);
                    ptx::tma_prefetch_3d(&tm_q, c * 64, nq0, nbh);
                    ptx::tma_prefetch_3d(&tm_do, c * 64, nq0, nbh);
                }
            }
            if (*abort_flag) {
                // The newest copy into each buffer is its newest phase.
                wait_bar(bar(L::B_RES_FULL), 0, ctl, SITE_BWD_DRAIN, false);
                for (int it = (issued_q > QS ? issued_q - QS : 0); it < issued_q; ++it)
                    wait_bar(bar(L::B_Q_FULL + it % QS), (it / QS) & 1, ctl, SITE_BWD_DRAIN, false);
                for (int it = (issued_do > DS ? issued_do - DS : 0); it < issued_do; ++it)
                    wait_bar(bar(L::B_DO_FULL + it % DS), (it / DS) & 1, ctl, SITE_BWD_DRAIN, false);
            }
        }
        __syncwarp();
    } else if (warp == BWD_MMA_WARP) {
        const uint32_t leader = elect_leader();
        constexpr uint32_t IDESC_SQ = ptx::idesc_f16(BF16, 128, 128, false, false);
        constexpr uint32_t IDESC_OD = ptx::idesc_f16(BF16, 128, D, false, true);
        const uint32_t d_s = tmem + BWD_TMEM_S, d_dp = tmem + BWD_TMEM_DP;
        const uint32_t d_dv = tmem + BWD_TMEM_A, d_dk = tmem + BWD_TMEM_B;
        auto stage_q = [&](int it) { return sbase + L::A_OFF + (it % QS) * L::TILE; };
        auto stage_do = [&](int it) { return sbase + L::B_OFF + (it % DS) * L::TILE; };
        auto issue_s = [&](int it) {  // S^T = K Q_i^T
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::mma_ss_if(leader, d_s, kmajor_desc(sbase + L::R0_OFF, kk), kmajor_desc(stage_q(it), kk), IDESC_SQ, kk > 0);
        };
        auto issue_dp = [&](int it) {  // dP^T = V dO_i^T
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::mma_ss_if(leader, d_dp, kmajor_desc(sbase + L::R1_OFF, kk), kmajor_desc(stage_do(it), kk), IDESC_SQ, kk > 0);
        };
        auto commit = [&](int b) { ptx::mma_commit_if(leader, bar(b)); };
        bool ok = n > 0 && wait_bar_warp(bar(L::B_RES_FULL), 0, ctl, SITE_BWD_MMA) &&
                  wait_bar_warp(bar(L::B_Q_FULL + 0), 0, ctl, SITE_BWD_MMA);
        if (ok) {
            ptx::tc_fence_after();
            issue_s(0);
            commit(L::B_S_FULL);
            ok = wait_bar_warp(bar(L::B_DO_FULL + 0), 0, ctl, SITE_BWD_MMA);
        }
        if (ok) {
            ptx::tc_fence_after();
            issue_dp(0);
            commit(L::B_DP_FULL);
        }
        for (int it = 0; ok && it < n; ++it) {
            // dV += P^T dO_i (P^T over the S^T columns), queries 0-63 as soon as they are stored
            for (int h = 0; h < 2 && ok; ++h) {
                if (!(ok = wait_bar_warp(bar(h == 0 ? L::B_P_HALF : L::B_P_FULL), it & 1, ctl, SITE_BWD_MMA)))
                    break;
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
                    ptx::mma_ts_if(leader, d_dv, d_s + kk * 8, mnmajor_desc(stage_do(it), kk), IDESC_OD,
                                    (it > 0 || kk > 0));
            }
            if (!ok) break;
            commit(L::B_DO_EMPTY + it % DS);  // dO_i's last reader
            if (it + 1 < n) {  // S^T of the next block may overwrite P^T now (MMAs run in order)
                if (!(ok = wait_bar_warp(bar(L::B_Q_FULL + (it + 1) % QS), ((it + 1) / QS) & 1, ctl, SITE_BWD_MMA))) break;
                ptx::tc_fence_after();
                issue_s(it + 1);
                commit(L::B_S_FULL);
            }
            // dK += dS^T Q_i (dS^T over the dP^T columns)
            if (!(ok = wait_bar_warp(bar(L::B_DS_FULL), it & 1, ctl, SITE_BWD_MMA))) break;
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                ptx::mma_ts_if(leader, d_dk, d_dp + kk * 8, mnmajor_desc(stage_q(it), kk), IDESC_OD, (it > 0 || kk > 0));
            commit(L::B_Q_EMPTY + it % QS);  // Q_i's last reader
            if (it + 1 < n) {
                if (!(ok = wait_bar_warp(bar(L::B_DO_FULL + (it + 1) % DS), ((it + 1) / DS) & 1, ctl, SITE_BWD_MMA))) break;
                ptx::tc_fence_after();
                issue_dp(it + 1);
                commit(L::B_DP_FULL);
            }
        }
        if (ok && n > 0) commit(L::B_MMA_DONE);
        if (*abort_flag) {
            commit(L::B_DRAIN);
            wait_bar(bar(L::B_DRAIN), 0, ctl, SITE_BWD_DRAIN, false);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- compute warps
        const int r = threadIdx.x;  // key row within the block
        const int kr = k0 + r;
        const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t s_cols = tmem + lanes + BWD_TMEM_S, dp_cols = tmem + lanes + BWD_TMEM_DP;
        // A zero scale would turn a hidden score's -inf into 0 * inf = NaN; a tiny one gives the
        // same weights. Hidden scores hold -inf (+inf under a negative scale), so 2^(s*c - L)
        // is 0 for them with no per-element test in the exponential loop.
        const float c = (p.scale_log2 == 0.f) ? 1e-30f : p.scale_log2;
        const uint32_t hidden = c < 0.f ? 0x7f800000u : 0xff800000u;
        bool ok = true;
        for (int it = 0; it < n; ++it) {
            const int i = i_begin + it;
            // lse2 landed with Q_i (before S^T(i) was computed), delta with dO_i (before dP^T(i)).
            const float* lse2 = reinterpret_cast<const float*>(smem + L::LSE_OFF + (it % QS) * L::VEC_BYTES);
            const float* dlt = reinterpret_cast<const float*>(smem + L::DELTA_OFF + (it % DS) * L::VEC_BYTES);
            if (!(ok = wait_bar_warp(bar(L::B_S_FULL), it & 1, ctl, SITE_BWD_COMPUTE))) break;
            ptx::tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int q = 0; q < 4; ++q) ptx::tmem_ld32(s_cols + q * 32, sr[q]);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 4; ++q) ptx::reg_fence(sr[q]);
            // P^T[r][col] = 2^(s*c - LSE2[col]); padded queries have LSE2 = +inf, so P = 0.
            // On the diagonal block a query before this key (q < k) does not see it.
            const bool diag = CAUSAL && (i == kb);
            if (diag) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (i * 128 + q * 32 + e < kr) sr[q][e] = hidden;
            }
            float pf[128];
            // P^T in two halves of 64 queries, each released to the dV product once stored.
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int qq = 0; qq < 2; ++qq)
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const int q = 2 * h + qq, col = q * 32 + e;
                        float x0, x1;
                        ffma2v(x0, x1, __uint_as_float(sr[q][e]), __uint_as_float(sr[q][e + 1]), c, c,
                                    -lse2[col], -lse2[col + 1]);
                        pf[col] = ptx::ex2(x0);
                        pf[col + 1] = ptx::ex2(x1);
                    }
                uint32_t pk[32];
#pragma unroll
                for (int w = 0; w < 32; ++w) pk[w] = pack2<BF16>(pf[h * 64 + 2 * w], pf[h * 64 + 2 * w + 1]);
                ptx::tmem_st32(s_cols + 32 * h, pk);
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(h == 0 ? L::B_P_HALF : L::B_P_FULL));
            }
            // dS^T[r][col] = P^T (dP^T - D[col]), written over the dP^T columns chunk by chunk
            // (chunk q of fp32 columns 32q.. becomes 16-bit pairs at 16q.., already read).
            if (!(ok = wait_bar_warp(bar(L::B_DP_FULL), it & 1, ctl, SITE_BWD_COMPUTE))) break;
            ptx::tc_fence_after();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t dr[32];
                ptx::tmem_ld32(dp_cols + q * 32, dr);
                ptx::tmem_wait_ld();
                ptx::reg_fence(dr);
                float ds[32];
#pragma unroll
                for (int e = 0; e < 32; e += 2)
                    fmulsub2(ds[e], ds[e + 1], pf[q * 32 + e], pf[q * 32 + e + 1],
                                  __uint_as_float(dr[e]), __uint_as_float(dr[e + 1]),
                                  dlt[q * 32 + e], dlt[q * 32 + e + 1]);
                uint32_t w[16];
                pack16<BF16>(ds, w);
                ptx::tmem_st16(dp_cols + q * 16, w);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(L::B_DS_FULL));
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(L::B_DO_EMPTY + it % DS));  // done with delta
        }
        // Epilogue: dV and scale * dK for this thread's key row.
        const size_t row_off = (static_cast<size_t>(bh) * p.nk + kr) * D * 2;
        const bool row_ok = kr >= p.nk || in_bounds(bh >= 0 && bh < p.bh && kr >= 0,
                                                    BOUNDS_BWD_DKDV,
                                                    static_cast<long long>(bh) * p.nk + kr);
        if (n == 0) {
            if (kr < p.nk && row_ok) {
                zero_row<D>(static_cast<uint8_t*>(p.dv) + row_off);
                zero_row<D>(static_cast<uint8_t*>(p.dk) + row_off);
            }
        } else if (ok && wait_bar_warp(bar(L::B_MMA_DONE), 0, ctl, SITE_BWD_COMPUTE)) {
            ptx::tc_fence_after();
            store_row<D, BF16>(tmem + lanes + BWD_TMEM_A, 1.f, static_cast<uint8_t*>(p.dv) + row_off, kr < p.nk && row_ok);
            store_row<D, BF16>(tmem + lanes + BWD_TMEM_B, p.scale, static_cast<uint8_t*>(p.dk) + row_off, kr < p.nk && row_ok);
        }
        ptx::tmem_wait_st();
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == BWD_MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------------------------
// dQ: one CTA per (slice, 128 queries); resident Q and dO; a ring of K tiles, a ring of V tiles
// ---------------------------------------------------------------------------------------------
// S_j = Q K_j^T alternates between two TMEM buffers (columns 0-127 and 384-511), so S_{j+1} and
// S_{j+2} are computed while the compute warps turn S_j and dP_j into dS_j. MMA order:
//   S_0, dP_0, S_1,  then per j: dP_{j+1}, dQ += dS_j K_j, S_{j+2} (over dS_j's buffer).
// K_j serves S_j and the dQ product of block j, so the K ring holds three tiles.
template <int D>
struct DqSmem {
    static constexpr int TILE = 128 * D * 2;
    static constexpr int K_STAGES = 3, V_STAGES = 2;
    static constexpr int Q_OFF = 0;
    static constexpr int DO_OFF = TILE;
    static constexpr int K_OFF = 2 * TILE;
    static constexpr int V_OFF = K_OFF + K_STAGES * TILE;
    static constexpr int BAR_OFF = V_OFF + V_STAGES * TILE;
    static constexpr int B_RES_FULL = 0;
    static constexpr int B_K_FULL = 1;                         // [K_STAGES]
    static constexpr int B_K_EMPTY = B_K_FULL + K_STAGES;      // [K_STAGES]
    static constexpr int B_V_FULL = B_K_EMPTY + K_STAGES;      // [V_STAGES]
    static constexpr int B_V_EMPTY = B_V_FULL + V_STAGES;      // [V_STAGES]
    static constexpr int B_S_FULL = B_V_EMPTY + V_STAGES;      // [2] per S buffer
    static constexpr int B_DP_FULL = B_S_FULL + 2;
    static constexpr int B_DS_FULL = B_DP_FULL + 1;
    static constexpr int B_MMA_DONE = B_DS_FULL + 1;
    static constexpr int B_DRAIN = B_MMA_DONE + 1;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int TMEM_SLOT_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int ABORT_OFF = TMEM_SLOT_OFF + 4;
    static constexpr int BYTES = ABORT_OFF + 4;
    static constexpr int ALLOC_BYTES = (BYTES + 1024 > 116 * 1024) ? BYTES + 1024 : 116 * 1024;
    static_assert(ALLOC_BYTES <= 232448, "shared memory budget");
};
constexpr uint32_t DQ_TMEM_S0 = 0, DQ_TMEM_DP = 128, DQ_TMEM_DQ = 256, DQ_TMEM_S1 = 384;

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdParams p) {
    using L = DqSmem<D>;
    constexpr int KS = L::K_STAGES, VS = L::V_STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = ptx::smem_u32(smem);
    auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * static_cast<uint32_t>(i); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::ABORT_OFF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::TMEM_SLOT_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int nkb = (p.nk + 127) / 128, nqb = (p.nq + 127) / 128;
    // Causal: the query blocks with the most key blocks (the last ones) first, across all slices,
    // so the last CTAs dispatched are the shortest (slice by slice, each slice's longest CTA came
    // last: 4-9 % slower); otherwise the CTAs of one slice are adjacent.
    const int bh = CAUSAL ? static_cast<int>(blockIdx.x % p.bh) : static_cast<int>(blockIdx.x / nqb);
    const int qb = CAUSAL ? nqb - 1 - static_cast<int>(blockIdx.x / p.bh) : static_cast<int>(blockIdx.x % nqb);
    const int q0 = qb * 128;
    const int n = CAUSAL ? min(nkb, qb + 1) : nkb;  // key blocks up to the diagonal

    const bool early = p.early_loads != 0;
    // Loads of the load lane: the resident Q and dO blocks; key block j of K and of V.
    auto load_res = [&]() {
        ptx::mbar_arrive_expect_tx(bar(L::B_RES_FULL), 2 * L::TILE);
        tma_tile<D>(sbase + L::Q_OFF, &tm_q, q0, bh, bar(L::B_RES_FULL));
        tma_tile<D>(sbase + L::DO_OFF, &tm_do, q0, bh, bar(L::B_RES_FULL));
    };
    auto load_k_blk = [&](int j) {
        const int ks = j % KS;
        ptx::mbar_arrive_expect_tx(bar(L::B_K_FULL + ks), L::TILE);
        tma_tile<D>(sbase + L::K_OFF + ks * L::TILE, &tm_k, j * 128, bh, bar(L::B_K_FULL + ks));
    };
    auto load_v_blk = [&](int j) {
        const int vs = j % VS;
        ptx::mbar_arrive_expect_tx(bar(L::B_V_FULL + vs), L::TILE);
        tma_tile<D>(sbase + L::V_OFF + vs * L::TILE, &tm_v, j * 128, bh, bar(L::B_V_FULL + vs));
    };
    if (threadIdx.x == (early ? BWD_LOAD_WARP * 32 : 0)) {
        *abort_flag = 0;
        ptx::mbar_init(bar(L::B_RES_FULL), 1);
        for (int s = 0; s < KS; ++s) {
            ptx::mbar_init(bar(L::B_K_FULL + s), 1);
            ptx::mbar_init(bar(L::B_K_EMPTY + s), 1);
        }
        for (int s = 0; s < VS; ++s) {
            ptx::mbar_init(bar(L::B_V_FULL + s), 1);
            ptx::mbar_init(bar(L::B_V_EMPTY + s), 1);
        }
        ptx::mbar_init(bar(L::B_S_FULL + 0), 1);
        ptx::mbar_init(bar(L::B_S_FULL + 1), 1);
        ptx::mbar_init(bar(L::B_DP_FULL), 1);
        ptx::mbar_init(bar(L::B_DS_FULL), 128);
        ptx::mbar_init(bar(L::B_MMA_DONE), 1);
        ptx::mbar_init(bar(L::B_DRAIN), 1);
        ptx::fence_barrier_init();
        ptx::fence_proxy_async_smem();
    }
    // Early mode: the load lane, which initialised the barriers just above, starts its loads
    // before the CTA barrier (this kernel reads nothing its predecessor in the stream writes).
    bool pre = false;
    if (early && threadIdx.x == BWD_LOAD_WARP * 32 && n > 0) {
        load_res();
        load_k_blk(0);
        load_v_blk(0);
        pre = true;
    }
    if (warp == BWD_MMA_WARP) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Ctl ctl{abort_flag, p.err, p.timeout_ns};
    auto s_buf = [](int j) { return (j & 1) ? DQ_TMEM_S1 : DQ_TMEM_S0; };

    if (warp == BWD_LOAD_WARP) {
        if (lane == 0) {
            if (!pre) load_res();
            int k_issued = pre ? 1 : 0, v_issued = pre ? 1 : 0;
            for (int j = pre ? 1 : 0; j < n; ++j) {
                const int ks = j % KS, vs = j % VS;
                if (!wait_bar(bar(L::B_K_EMPTY + ks), ((j / KS) & 1) ^ 1, ctl, SITE_BWD_LOAD)) break;
                load_k_blk(j);
                k_issued = j + 1;
                if (!wait_bar(bar(L::B_V_EMPTY + vs), ((j / VS) & 1) ^ 1, ctl, SITE_BWD_LOAD)) break;
                load_v_blk(j);
                v_issued = j + 1;
            }
            // The CTA one wave later: its Q and dO blocks and its first K and V blocks.
            const int nb = static_cast<int>(blockIdx.x) + p.next_prefetch_stride;
            if (p.next_prefetch_stride > 0 && nb < static_cast<int>(gridDim.x) && !*abort_flag) {
                const int nbh = CAUSAL ? nb % p.bh : nb / nqb;
                const int nq0 = (CAUSAL ? nqb - 1 - nb / p.bh : nb % nqb) * 128;
                for (int c = 0; c < D / 64; ++c) {
                    ptx::tma_prefetch_3d(&tm_q, c * 64, nq0, nbh);
                    ptx::tma_prefetch_3d(&tm_do, c * 64, nq0, nbh);
                    ptx::tma_prefetch_3d(&tm_k, c * 64, 0, nbh);
                    ptx::tma_prefetch_3d(&tm_v, c * 64, 0, nbh);
                }
            }
            if (*abort_flag) {
                // Drain: the newest copy into each stage is its barrier's newest phase.
                wait_bar(bar(L::B_RES_FULL), 0, ctl, SITE_BWD_DRAIN, false);
                for (int j = (k_issued > KS ? k_issued - KS : 0); j < k_issued; ++j)
                    wait_bar(bar(L::B_K_FULL + j % KS), (j / KS) & 1, ctl, SITE_BWD_DRAIN, false);
                for (int j = (v_issued > VS ? v_issued - VS : 0); j < v_issued; ++j)
                    wait_bar(bar(L::B_V_FULL + j % VS), (j / VS) & 1, ctl, SITE_BWD_DRAIN, false);
            }
        }
        __syncwarp();
    } else if (warp == BWD_MMA_WARP) {
        const uint32_t leader = elect_leader();
        constexpr uint32_t IDESC_SQ = ptx::idesc_f16(BF16, 128, 128, false, false);
        constexpr uint32_t IDESC_OD = ptx::idesc_f16(BF16, 128, D, false, true);
        const uint32_t d_dp = tmem + DQ_TMEM_DP, d_dq = tmem + DQ_TMEM_DQ;
        auto commit = [&](int b) { ptx::mma_commit_if(leader, bar(b)); };
        auto k_tile = [&](int j) { return sbase + L::K_OFF + (j % KS) * L::TILE; };
        auto v_tile = [&](int j) { return sbase + L::V_OFF + (j % VS) * L::TILE; };
        // S_j = Q K_j^T into the buffer of block j.
        auto issue_s = [&](int j) -> bool {
            if (!wait_bar_warp(bar(L::B_K_FULL + j % KS), (j / KS) & 1, ctl, SITE_BWD_MMA)) return false;
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::mma_ss_if(leader, tmem + s_buf(j), kmajor_desc(sbase + L::Q_OFF, kk),
                                kmajor_desc(k_tile(j), kk), IDESC_SQ, kk > 0);
            commit(L::B_S_FULL + (j & 1));
            return true;
        };
        // dP_j = dO V_j^T; V_j is then free.
        auto issue_dp = [&](int j) -> bool {
            if (!wait_bar_warp(bar(L::B_V_FULL + j % VS), (j / VS) & 1, ctl, SITE_BWD_MMA)) return false;
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::mma_ss_if(leader, d_dp, kmajor_desc(sbase + L::DO_OFF, kk), kmajor_desc(v_tile(j), kk),
                                IDESC_SQ, kk > 0);
            commit(L::B_DP_FULL);
            commit(L::B_V_EMPTY + j % VS);
            return true;
        };
        bool ok = wait_bar_warp(bar(L::B_RES_FULL), 0, ctl, SITE_BWD_MMA);
        ok = ok && issue_s(0) && issue_dp(0) && (n < 2 || issue_s(1));
        for (int j = 0; ok && j < n; ++j) {
            if (!(ok = wait_bar_warp(bar(L::B_DS_FULL), j & 1, ctl, SITE_BWD_MMA))) break;
            // dP_{j+1} first: the compute warps are done with dP_j, and dS_{j+1} then overlaps
            // the dQ product of block j instead of waiting behind it.
            if (j + 1 < n && !(ok = issue_dp(j + 1))) break;
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // dQ += dS_j K_j (dS_j over its S buffer)
                ptx::mma_ts_if(leader, d_dq, tmem + s_buf(j) + kk * 8, mnmajor_desc(k_tile(j), kk), IDESC_OD,
                                (j > 0 || kk > 0));
            commit(L::B_K_EMPTY + j % KS);
            if (j + 2 < n && !(ok = issue_s(j + 2))) break;
        }
        if (ok) commit(L::B_MMA_DONE);
        if (*abort_flag) {
            commit(L::B_DRAIN);
            wait_bar(bar(L::B_DRAIN), 0, ctl, SITE_BWD_DRAIN, false);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- compute warps
        const int r = threadIdx.x;
        const int row = q0 + r;
        const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t dp_cols = tmem + lanes + DQ_TMEM_DP;
        // A zero scale would turn a hidden score's -inf into 0 * inf = NaN; a tiny one gives the
        // same weights. Hidden scores hold -inf (+inf under a negative scale), so 2^(s*c - L)
        // is 0 for them with no per-element test in the exponential loop.
        const float c = (p.scale_log2 == 0.f) ? 1e-30f : p.scale_log2;
        const uint32_t hidden = c < 0.f ? 0x7f800000u : 0xff800000u;
        const size_t vo = static_cast<size_t>(bh) * p.nq_pad + row;  // row < nq_pad always
        const float lse2 = p.lse2[vo], dlt = p.delta[vo];
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const uint32_t s_cols = tmem + lanes + s_buf(j);
            if (!(ok = wait_bar_warp(bar(L::B_S_FULL + (j & 1)), (j >> 1) & 1, ctl, SITE_BWD_COMPUTE))) break;
            ptx::tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int q = 0; q < 4; ++q) ptx::tmem_ld32(s_cols + q * 32, sr[q]);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 4; ++q) ptx::reg_fence(sr[q]);
            // P = 2^(s*c - LSE2); keys past Nk and (causal) keys after the query get 0.
            const int k0 = j * 128;
            int lim = p.nk - k0;
            if constexpr (CAUSAL) lim = min(lim, row + 1 - k0);
            if (lim < 128) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (q * 32 + e >= lim) sr[q][e] = hidden;
            }
            float pf[128];
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float x0, x1;
                    ptx::ffma2(x0, x1, __uint_as_float(sr[q][e]), __uint_as_float(sr[q][e + 1]), c, -lse2);
                    pf[q * 32 + e] = ptx::ex2(x0);
                    pf[q * 32 + e + 1] = ptx::ex2(x1);
                }
            if (!(ok = wait_bar_warp(bar(L::B_DP_FULL), j & 1, ctl, SITE_BWD_COMPUTE))) break;
            ptx::tc_fence_after();
            // dS = P (dP - D), written over this block's S buffer (all of S is in registers). dP
            // comes in two loads of 64 columns, each waited for once.
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t dr[2][32];
                ptx::tmem_ld32(dp_cols + (2 * h) * 32, dr[0]);
                ptx::tmem_ld32(dp_cols + (2 * h + 1) * 32, dr[1]);
                ptx::tmem_wait_ld();
                ptx::reg_fence(dr[0]);
                ptx::reg_fence(dr[1]);
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    const int q = 2 * h + qq;
                    float ds[32];
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        fmulsub2(ds[e], ds[e + 1], pf[q * 32 + e], pf[q * 32 + e + 1],
                                      __uint_as_float(dr[qq][e]), __uint_as_float(dr[qq][e + 1]), dlt, dlt);
                    uint32_t w[16];
                    pack16<BF16>(ds, w);
                    ptx::tmem_st16(s_cols + q * 16, w);
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(L::B_DS_FULL));
        }
        if (ok && n > 0 && wait_bar_warp(bar(L::B_MMA_DONE), 0, ctl, SITE_BWD_COMPUTE)) {
            ptx::tc_fence_after();
            store_row<D, BF16>(tmem + lanes + DQ_TMEM_DQ, p.scale,
                               static_cast<uint8_t*>(p.dq) + (static_cast<size_t>(bh) * p.nq + row) * D * 2,
                               row < p.nq && in_bounds(bh >= 0 && bh < p.bh && row >= 0,
                                                       BOUNDS_BWD_DQ,
                                                       static_cast<long long>(bh) * p.nq + row));
        }
        ptx::tmem_wait_st();
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == BWD_MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
    // This grid does not wait for the dK/dV kernel it was launched after (it reads nothing that
    // kernel writes), but it completes only after it, so that work later in the stream that
    // waits for this grid also sees dK and dV: one CTA, the last one, waits for it before exiting.
    // Waiting in every CTA would hold SMs that later CTAs of this grid could use.
    if (blockIdx.x == gridDim.x - 1) asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace fa
