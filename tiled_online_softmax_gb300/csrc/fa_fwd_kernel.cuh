// fa_fwd_kernel.cuh -- the sm_103a attention forward kernel (tiled online softmax).
//
// Work unit: 256 query rows of one (batch, head) slice, as two tiles of BM = 128 rows that share
// every K/V tile the CTA loads; keys stream past in tiles of BN = 128 ("11. Fusion, recompute,
// and flash attention", section 11.9: one thread block per block of query rows, the query block
// loaded once, key blocks looped over). For query tile t and key tile j:
//
//   S_t = Q_t K_j^T                     tcgen05 MMA, fp32 accumulator in tensor memory (TMEM)
//   m_new = max(m, rowmax S_t * c)      c = scale * log2(e): every exponential is a bare exp2
//   corr  = 2^(m - m_new)               (same chapter, section 11.7, base 2 with log2 e folded
//   P_t   = 2^(S_t * c - m_new)          into the scale)
//   l     = l * corr + rowsum P_t
//   O_t   = O_t * corr + P_t V_j        rescale of O_t in TMEM, then an MMA with P_t from TMEM
//
// and after the last key tile O_t / l is written once ("Flash Attention 2", "Write the data back
// to HBM"). The recurrence is section 11.6 "Online softmax" one key block at a time ("Flash
// Attention 2", "Overview of the algorithm"; phobos "Attention", `online_softmax`). The maximum
// is updated lazily: while a row's new maximum exceeds its reference maximum by at most a
// threshold (log2 units: 32 for bf16, at most 15 for fp16), the reference is kept and nothing is
// rescaled (the conditional rescaling of ithelp article 10405336, FlashAttention 保留三個狀態);
// l and O share the reference, so O / l is unchanged and P stays <= 2^threshold.
//
// Warp roles (384 threads, registers rebalanced with setmaxnreg):
//   warpgroup 0 (warps 0-3)  softmax of query tile 0: thread r owns row r (TMEM lane r), so row
//                            max and sum need no shuffles. When a row of the warp moves its
//                            reference max, the warp also rescales its rows of O_0 in TMEM.
//   warpgroup 1 (warps 4-7)  softmax of query tile 1.
//                            After its key loop each of them writes its tile: O_t / l, rounded,
//                            staged in shared memory and stored by TMA.
//   warp 8                   MMA issuer (one elected lane issues, as predicated instructions
//                            the whole warp runs) and TMEM owner.
//   warp 9                   TMA producer (one lane): Q_0, K_0, Q_1, V_0, then K and V tiles
//                            through rings of stages.
//   warps 10-11              idle.
// The grid is launched as a programmatic dependent of the stream's previous kernel; its set-up
// may overlap that kernel's end, and no global memory is read or written before
// griddepcontrol.wait (the first wave of a causal launch issues L2 prefetch hints for its first
// tiles before it, which move no data into the SM). The TMA lane initialises the barriers and
// issues the first Q and K loads before the CTA-wide barrier; once its own loads are issued it
// prefetches into L2 the first tiles of the CTA one wave later.
// D = 128: the MMA warp issues, per key tile j: PV_0(j) in two halves (keys 0-63 as soon as the
// softmax releases them, then 64-127), S_0(j+1), PV_1(j) likewise, S_1(j+1). While one tile's
// softmax runs, the tensor cores work on the other tile's products; each tile's S_t(j+1) waits
// for PV_t(j), because it overwrites P_t(j).
// D = 64: the two O accumulators leave room for a third S/P buffer, and the S products of both
// tiles rotate through the three (the k-th S product of the CTA, in issue order, goes to buffer
// k mod 3). The MMA warp issues PV of product k - 3, which frees its buffer, then S product k. A
// tile's next S product no longer waits for the PV product of its current one, so it can be
// computed while the tile's softmax still works on the current step.
//
// Tensor memory (512 columns x 128 lanes of 32 bit):
//   D = 128: [0,128) S_0 (fp32), its first 64 columns take P_0 (16-bit pairs) once S_0 is read;
//            [128,256) S_1 / P_1;  [256,384) O_0;  [384,512) O_1.
//   D = 64:  [0,128), [128,256), [256,384) the three S / P buffers;  [384,448) O_0;  [448,512) O_1.
//
// Masking: a key j >= Nk (partial last tile, phobos "Attention", `attention`) or, under causal
// masking, a key after the query (phobos "Causal attention") is left out of the row max and gets
// weight 0; key tiles entirely after a query tile's last row are never computed for that tile.
//
// Every wait is bounded: past the time limit the waiting thread records a site code in the
// device error word, raises the CTA's abort flag, and every role winds down (waiting, bounded
// again, for its own in-flight copies and MMAs) before TMEM is freed and the CTA exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "fa_bounds.cuh"
#include "fa_rope_kernel.cuh"
#include "sm103_ptx.cuh"

namespace fa {

constexpr int BM = 128;              // query rows per tile = TMEM lanes
constexpr int BN = 128;              // keys per tile
constexpr int Q_TILES = 2;           // query tiles per CTA (one work unit = 256 rows)
constexpr int UNIT_ROWS = BM * Q_TILES;
constexpr int NUM_THREADS = 384;
constexpr int MMA_WARP = 8;
constexpr int LOAD_WARP = 9;
constexpr uint32_t TMEM_COLS = 512;
// Three S / P buffers rotating between the two tiles (D = 64), or one per tile (D = 128).
template <int D>
constexpr bool S_RING = (D == 64);
template <int D>
__host__ __device__ constexpr uint32_t tmem_o(int t) {
    return S_RING<D> ? 384u + 64u * static_cast<uint32_t>(t) : (t ? 384u : 256u);
}
// Number of S_t(j) in the order the MMA warp issues a CTA's S products: the two tiles alternate
// while both have key tiles left, then tile 1 alone (n0 = tile 0's key tiles <= tile 1's: its
// rows come first). Its TMEM buffer: tmem_s_buf.
__host__ __device__ constexpr int s_seq(int t, int j, int n0) { return j < n0 ? 2 * j + t : n0 + j; }
template <int D>
__host__ __device__ constexpr uint32_t tmem_s_buf(int t, int j, int n0) {
    return S_RING<D> ? 128u * static_cast<uint32_t>(s_seq(t, j, n0) % 3) : (t ? 128u : 0u);
}

// Registers per thread after rebalancing. The launch gives each of the 384 threads 168 (the
// most that fits 65536); the two softmax warpgroups then take 216 each, the MMA/TMA warpgroup
// keeps 72.
constexpr uint32_t REG_LAUNCH = 168, REG_SOFTMAX = 216, REG_MISC = 72;
static_assert(NUM_THREADS * REG_LAUNCH <= 65536, "launch register file");
static_assert(2 * 128 * REG_SOFTMAX + 128 * REG_MISC <= NUM_THREADS * REG_LAUNCH,
              "setmaxnreg split exceeds the launch's register file");

// Wait-site codes written to the device error word (first timeout wins).
enum WaitSite : int {
    SITE_LOAD_K_EMPTY = 1,
    SITE_LOAD_V_EMPTY = 2,
    SITE_MMA_Q_FULL = 3,
    SITE_MMA_K_FULL = 4,
    SITE_MMA_P_FULL = 5,
    SITE_MMA_V_FULL = 6,
    SITE_SOFTMAX_S_FULL = 7,
    SITE_SOFTMAX_O_DONE = 8,
    SITE_EPI_O_READY = 9,
    SITE_DRAIN = 10,
    SITE_EPI_O_STAGED = 14,
    SITE_ROPE_Q_FULL = 15,
    SITE_SELFTEST = 30,   // fa_wait_selftest: a barrier that nothing arrives on
};

// Floor of the time limit of drain waits (for copies and MMAs this CTA started, which always
// complete): a short limit for the ordinary waits never lets a CTA exit with copies in flight.
constexpr unsigned long long DRAIN_FLOOR_NS = 1000000000ull;
// Longest sleep of one try inside a bounded wait (the waiting thread wakes as soon as the phase
// completes); the time limit is checked every 32 tries.
constexpr uint32_t WAIT_SLEEP_NS = 2000;

struct Params {
    void* o;                   // output [bh][nq][D]
    float* lse;                // optional log-sum-exp output [bh][nq] (natural log), or null
    int* err;                  // device error word (site code of the first timeout)
    int bh;                    // B * H
    int nq, nk;
    int num_units;             // ceil(nq / 256)
    // Split over keys (non-causal only). Units are numbered bh * num_units + u. CTAs below
    // split_begin run one whole unit each; the units from split_begin on run as num_splits CTAs
    // each, CTA (unit, s) covering key tiles [s * kv_tiles_per_split, ...) and writing its
    // unnormalised state instead of O, for split unit t = unit - split_begin and its row r:
    //   o_part [num_splits][t][split_rows][D] fp32, ml_part [num_splits][t][split_rows][2]
    //   fp32 (m in log2 units of the scaled scores, l relative to it), split_rows = min(256, nq).
    int num_splits;
    int kv_tiles_per_split;
    int split_begin;
    int split_units;
    float* o_part;
    float* ml_part;
    float scale_log2;          // scale * log2(e)
    float rescale_threshold;   // lazy-rescale threshold, log2 units (0 = rescale on every rise)
    unsigned long long timeout_ns;
    // Rotary embedding of Q inside the kernel (null: none): angle tables [nq][D/2] fp32 of the
    // query rows, and the pair form (0 rotate-half, 1 interleaved pairs).
    const float* rope_cos;
    const float* rope_sin;
    int rope_form;
    // fp32 output (null: none): O / l written unrounded as fp32 [bh][nq][D] instead of the
    // 16-bit O, to check the arithmetic apart from the output rounding.
    float* o_f32;
    // CTAs below this index (the first wave) prefetch their first tiles into L2 before waiting
    // for the previous kernel (0: none).
    int prefetch_ctas;
    // After issuing its last loads, each CTA prefetches into L2 the first tiles of CTA
    // blockIdx.x + next_prefetch_stride, one wave later (0: none).
    int next_prefetch_stride;
    // The TMA lane initialises the barriers itself and issues the first Q and K loads before the
    // CTA-wide barrier, overlapping the rest of the set-up (0: after it, as the other roles).
    int early_loads;
};

template <int D>
struct Smem {
    static constexpr int STAGES = (D == 64) ? 4 : 2;
    static constexpr int COL_BLOCKS = D / 64;            // 128-byte (64-element) column blocks
    static constexpr int Q_TILE_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2;          // one K or V tile
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + Q_TILES * Q_TILE_BYTES;
    static constexpr int V_OFF = K_OFF + STAGES * KV_BYTES;
    static constexpr int BAR_OFF = V_OFF + STAGES * KV_BYTES;
    // barrier indices
    static constexpr int B_Q_FULL = 0;                          // [2]
    static constexpr int B_K_FULL = B_Q_FULL + Q_TILES;         // [STAGES]
    static constexpr int B_K_EMPTY = B_K_FULL + STAGES;
    static constexpr int B_V_FULL = B_K_EMPTY + STAGES;
    static constexpr int B_V_EMPTY = B_V_FULL + STAGES;
    // The per-step hand-offs use one barrier per tile, or with the S ring one per buffer: a
    // tile's softmax may then run up to two steps ahead of the PV product that consumes its P,
    // but a buffer is reused only after the PV of its previous product has been issued, so each
    // barrier completes at most one phase ahead of its waiter.
    static constexpr int HAND = S_RING<D> ? 3 : Q_TILES;
    static constexpr int B_S_FULL = B_V_EMPTY + STAGES;         // [HAND] MMA -> softmax
    static constexpr int B_P_HALF = B_S_FULL + HAND;            // [HAND] softmax -> MMA (keys 0-63)
    static constexpr int B_P_FULL = B_P_HALF + HAND;            // [HAND] softmax -> MMA (keys 64-127)
    static constexpr int B_O_DONE = B_P_FULL + HAND;            // [2] (S ring) PV_t(j) complete
    static constexpr int B_O_READY = B_O_DONE + (S_RING<D> ? Q_TILES : 0);  // [2] MMA -> epilogue
    static constexpr int B_O_STAGED = B_O_READY + Q_TILES;      // [2] O_t in smem (4 warps)
    static constexpr int B_Q_ROT = B_O_STAGED + Q_TILES;        // [2] Q_t rotated (8 warps)
    static constexpr int B_DRAIN = B_Q_ROT + Q_TILES;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int TMEM_SLOT_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int ABORT_OFF = TMEM_SLOT_OFF + 4;
    static constexpr int BYTES = ABORT_OFF + 4;
    static constexpr int ALLOC_BYTES = BYTES + 1024;            // slack for 1024-byte alignment
    static_assert(ALLOC_BYTES <= 232448, "shared memory budget");
    // More than half an SM's shared memory, so two CTAs never share an SM: each holds all 512
    // TMEM columns, and a second one would stall in tcgen05.alloc.
    static_assert(ALLOC_BYTES > 116 * 1024, "one CTA per SM");
    // Hand-off barrier of tile t's key step j (base: B_S_FULL, B_P_HALF or B_P_FULL; n0: tile
    // 0's key tiles), and the phase parity that step completes on it.
    __device__ static constexpr int hand(int base, int t, int j, int n0) {
        return base + (S_RING<D> ? s_seq(t, j, n0) % 3 : t);
    }
    __device__ static constexpr uint32_t hand_parity(int t, int j, int n0) {
        return static_cast<uint32_t>(S_RING<D> ? (s_seq(t, j, n0) / 3) & 1 : j & 1);
    }
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
    const uint64_t limit =
        honor_abort || ctl.timeout_ns >= DRAIN_FLOOR_NS ? ctl.timeout_ns : DRAIN_FLOOR_NS;
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait_sleep(bar, parity, WAIT_SLEEP_NS)) return true;
        if ((it & 31u) == 0) {
            if (honor_abort && *ctl.abort) return false;
            if (ptx::globaltimer_ns() - t0 > limit) {
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

// One warp waits, through wait_bar, on an mbarrier that expects one arrival which never comes:
// the wait runs out after timeout_ns and leaves SITE_SELFTEST in the error word. It exercises
// the timeout path of every kernel's waits without a real stall.
__global__ void __launch_bounds__(32) fa_wait_selftest_kernel(int* err, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t mbar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        ptx::mbar_init(static_cast<uint32_t>(__cvta_generic_to_shared(&mbar)), 1);
        ptx::fence_barrier_init();
    }
    __syncwarp();
    const Ctl ctl{&abort_flag, err, timeout_ns};
    wait_bar_warp(static_cast<uint32_t>(__cvta_generic_to_shared(&mbar)), 0, ctl, SITE_SELFTEST);
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

// The two 16-bit halves of a 32-bit word as fp32 (low half first).
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t u) {
    if constexpr (BF16) {
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
    } else {
        return __half22float2(*reinterpret_cast<const __half2*>(&u));
    }
}

// ---------------------------------------------------------------------------------------------
// epilogue of query tile t (its softmax warpgroup, after the key loop): O_t / l, rounded to the
// 16-bit type, one row per thread
// ---------------------------------------------------------------------------------------------
template <int D, bool BF16>
__device__ __forceinline__ void epilogue(int t, uint32_t tmem, uint32_t sbase, const Params& p,
                                         const Ctl& ctl, int bh, int q0, int split, float l,
                                         float m_ref, const CUtensorMap* tm_o) {
    using L = Smem<D>;
    auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * static_cast<uint32_t>(i); };
    const int r = threadIdx.x & 127;
    const int warp = threadIdx.x >> 5;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t o_cols = tmem + lane_base + tmem_o<D>(t);
    const int row = q0 + t * BM + r;
    if (!wait_bar_warp(bar(L::B_O_READY + t), 0, ctl, SITE_EPI_O_READY)) return;
    ptx::tc_fence_after();
    if (split >= 0) {
        // Partial state over this CTA's keys, merged later (split over keys).
        const int split_rows = min(UNIT_ROWS, p.nq);
        const int tu = bh * p.num_units + q0 / UNIT_ROWS - p.split_begin;
        const size_t prow =
            (static_cast<size_t>(split) * p.split_units + tu) * split_rows + (row - q0);
        const bool part_ok =
            row >= p.nq || in_bounds(split < p.num_splits && tu >= 0 && tu < p.split_units &&
                                         row - q0 < split_rows,
                                     BOUNDS_FWD_PART, static_cast<long long>(prow));
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            ptx::tmem_ld32(o_cols + q * 32, o);
            ptx::tmem_wait_ld();
            ptx::reg_fence(o);
            if (row < p.nq && part_ok) {
                uint4* dst = reinterpret_cast<uint4*>(p.o_part + prow * D + q * 32);
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    dst[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
            }
        }
        if (row < p.nq && part_ok) reinterpret_cast<float2*>(p.ml_part)[prow] = make_float2(m_ref, l);
        return;
    }
    if (p.lse != nullptr && row < p.nq &&
        in_bounds(bh >= 0 && bh < p.bh, BOUNDS_FWD_LSE, static_cast<long long>(bh) * p.nq + row)) {
        // L = m + log l in natural-log units ("Flash Attention 2", "Write the data back to
        // HBM"): the kernel's m and l are in base 2 relative to the reference maximum.
        p.lse[static_cast<size_t>(bh) * p.nq + row] = (m_ref + __log2f(l)) * 0.6931471805599453f;
    }
    if (p.o_f32 != nullptr) {
        // O_t / l in fp32, one row per thread, unrounded.
        const float inv_l32 = (l > 0.f) ? 1.f / l : 0.f;
        const bool keep = row < p.nq && in_bounds(bh >= 0 && bh < p.bh, BOUNDS_FWD_O,
                                                  static_cast<long long>(bh) * p.nq + row);
        float* dst_row = p.o_f32 + (static_cast<size_t>(bh) * p.nq + row) * D;
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            ptx::tmem_ld32(o_cols + q * 32, o);
            ptx::tmem_wait_ld();
            ptx::reg_fence(o);
            if (keep) {
                float4* dst = reinterpret_cast<float4*>(dst_row + q * 32);
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv_l32,
                                         __uint_as_float(o[4 * v + 1]) * inv_l32,
                                         __uint_as_float(o[4 * v + 2]) * inv_l32,
                                         __uint_as_float(o[4 * v + 3]) * inv_l32);
            }
        }
        return;
    }
    // O_t / l, rounded, staged in shared memory over Q_t (whose last reader, S_t of the last key
    // tile, finished before O_READY_t) in the 128-byte-swizzled layout of the tensor map, then
    // written by TMA: whole 128-byte row segments instead of one 16-byte store per row.
    const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
    const uint32_t stage = sbase + L::Q_OFF + t * L::Q_TILE_BYTES;
    // All of the row's O at once (D columns), then one wait.
    uint32_t o[D / 32][32];
    if constexpr (D == 128) {
        ptx::tmem_ld128(o_cols, o);
    } else {
#pragma unroll
        for (int q = 0; q < D / 32; ++q) ptx::tmem_ld32(o_cols + q * 32, o[q]);
    }
    ptx::tmem_wait_ld();
#pragma unroll
    for (int q = 0; q < D / 32; ++q) ptx::reg_fence(o[q]);
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            packed[i] = pack2<BF16>(__uint_as_float(o[q][2 * i]) * inv_l,
                                    __uint_as_float(o[q][2 * i + 1]) * inv_l);
        // 32 columns = 4 chunks of 16 bytes in column block q / 2, chunks 4 (q % 2) + v of the
        // row; chunk c of row r sits at chunk position c ^ (r % 8).
        const uint32_t row_base = stage + (q / 2) * (BM * 128) + r * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint32_t c = (q % 2) * 4 + v;
            ptx::st_shared_v4(row_base + ((c ^ (r & 7)) << 4), packed[4 * v], packed[4 * v + 1],
                              packed[4 * v + 2], packed[4 * v + 3]);
        }
    }
    ptx::fence_proxy_async_smem();  // the TMA store reads what these threads wrote
    __syncwarp();
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(bar(L::B_O_STAGED + t));
    if (r == 0) {
        if (!wait_bar(bar(L::B_O_STAGED + t), 0, ctl, SITE_EPI_O_STAGED)) return;
        // The tensor map clips rows past Nq (a decoding shape's second tile is wholly past it);
        // the unit itself must start inside the tensor.
        if (!in_bounds(bh >= 0 && bh < p.bh && q0 >= 0 && q0 < p.nq, BOUNDS_FWD_O,
                       static_cast<long long>(bh) * p.nq + q0))
            return;
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
            ptx::tma_store_3d(tm_o, stage + cb * (BM * 128), cb * 64, q0 + t * BM, bh);
        ptx::bulk_commit_group();
        ptx::bulk_wait_group_read0();  // shared memory stays allocated until the copy has read it
    }
}

// ---------------------------------------------------------------------------------------------
// rotary embedding of the Q tiles in shared memory ("Attention", phobos stdlib docs, "Rotary
// position embeddings"), by both softmax warpgroups before their key loops. The work of a tile is
// 128 rows x D/8 items of 4 pairs (pairs 4g .. 4g+3 of a row, angles cos/sin[row][4g .. 4g+4));
// thread x of the 256 takes items x, x + 256, ..., so consecutive lanes take consecutive items of
// one row: their angle loads are coalesced, and their shared-memory accesses cover whole 128-byte
// rows. Tile 0 is rotated first, then tile 1; after each, every warp signals B_Q_ROT_t, which the
// MMA warp waits on instead of the load. The producer loads both Q tiles before K_0 in this mode,
// so the rotation overlaps K_0's load. All angles are loaded before the first wait. Rows past Nq
// (zero fill, never stored) are left as they are.
// ---------------------------------------------------------------------------------------------
template <int D, bool BF16>
__device__ __forceinline__ bool rotate_q(uint32_t sbase, const Params& p, const Ctl& ctl, int q0) {
    using L = Smem<D>;
    constexpr int ITEMS_PER_ROW = D / 8;                   // items of 4 pairs per row
    constexpr int PER_THREAD = BM * ITEMS_PER_ROW / 256;   // items per thread and tile
    const int x = threadIdx.x;                             // 0..255
    float4 cs[Q_TILES][PER_THREAD], sn[Q_TILES][PER_THREAD];
#pragma unroll
    for (int t = 0; t < Q_TILES; ++t)
#pragma unroll
        for (int k = 0; k < PER_THREAD; ++k) {
            const int item = k * 256 + x, r = item / ITEMS_PER_ROW, g = item % ITEMS_PER_ROW;
            const int row = q0 + t * BM + r;
            if (row < p.nq) {
                const size_t off = static_cast<size_t>(row) * (D / 2) + 4 * g;
                cs[t][k] = __ldg(reinterpret_cast<const float4*>(p.rope_cos + off));
                sn[t][k] = __ldg(reinterpret_cast<const float4*>(p.rope_sin + off));
            }
        }
#pragma unroll
    for (int t = 0; t < Q_TILES; ++t) {
        const uint32_t q_full = sbase + L::BAR_OFF + 8u * static_cast<uint32_t>(L::B_Q_FULL + t);
        if (!wait_bar_warp(q_full, 0, ctl, SITE_ROPE_Q_FULL)) return false;
        const uint32_t tile = sbase + L::Q_OFF + t * L::Q_TILE_BYTES;
#pragma unroll
        for (int k = 0; k < PER_THREAD; ++k) {
            const int item = k * 256 + x, r = item / ITEMS_PER_ROW, g = item % ITEMS_PER_ROW;
            if (q0 + t * BM + r >= p.nq) continue;
            // Logical 16-byte chunk c (elements 8c .. 8c+7) of row r: column block c / 8,
            // swizzled position (c % 8) ^ (r % 8) within the row's 128 bytes.
            auto chunk = [&](int c) {
                return tile + (c / 8) * (BM * 128) + r * 128 +
                       ((static_cast<uint32_t>(c % 8) ^ (r & 7)) << 4);
            };
            const float c4[4] = {cs[t][k].x, cs[t][k].y, cs[t][k].z, cs[t][k].w};
            const float s4[4] = {sn[t][k].x, sn[t][k].y, sn[t][k].z, sn[t][k].w};
            if (p.rope_form == 0) {
                // pair i = (x_i, x_{i+D/2}): elements 4g .. 4g+3 (half g % 2 of chunk g / 2) with
                // the same 8 bytes of chunk g / 2 + D/16
                const uint32_t a_addr = chunk(g / 2) + (g % 2) * 8;
                const uint32_t b_addr = chunk(g / 2 + D / 16) + (g % 2) * 8;
                const uint2 a = ptx::ld_shared_v2(a_addr), b = ptx::ld_shared_v2(b_addr);
                const uint32_t av[2] = {a.x, a.y}, bv[2] = {b.x, b.y};
                uint32_t ao[2], bo[2];
                rope_half4<BF16>(av, bv, c4, s4, ao, bo);
                ptx::st_shared_v2(a_addr, ao[0], ao[1]);
                ptx::st_shared_v2(b_addr, bo[0], bo[1]);
            } else {
                // pair i = (x_{2i}, x_{2i+1}): pairs 4g .. 4g+3 are chunk g
                const uint4 v = ptx::ld_shared_v4(chunk(g));
                const uint32_t xv[4] = {v.x, v.y, v.z, v.w};
                uint32_t y[4];
                rope_pairs_n<BF16, 4>(xv, c4, s4, y);
                ptx::st_shared_v4(chunk(g), y[0], y[1], y[2], y[3]);
            }
        }
        ptx::fence_proxy_async_smem();  // the S products read the tile through the async proxy
        __syncwarp();
        if ((threadIdx.x & 31) == 0)
            ptx::mbar_arrive(sbase + L::BAR_OFF + 8u * static_cast<uint32_t>(L::B_Q_ROT + t));
    }
    return true;
}

// ---------------------------------------------------------------------------------------------
// softmax of one query tile (warpgroup t)
// ---------------------------------------------------------------------------------------------
template <int D, bool BF16, bool CAUSAL>
__device__ __forceinline__ void softmax_role(int t, uint32_t tmem, uint32_t sbase,
                                             const Params& p, const Ctl& ctl, int bh, int q0,
                                             int split, int kv0, int n_tiles, int n_first,
                                             const CUtensorMap* tm_o) {
    using L = Smem<D>;
    auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * static_cast<uint32_t>(i); };
    const int r = threadIdx.x & 127;          // row within the tile = TMEM lane
    const int warp = threadIdx.x >> 5;
    const int q_tile0 = q0 + t * BM;
    const int row = q_tile0 + r;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t o_cols = tmem + lane_base + tmem_o<D>(t);
    // A zero scale would turn the -inf of a hidden score into 0 * inf = NaN; a tiny positive
    // scale gives the same weights (every visible score maps to 2^0 = 1) and keeps -inf -> 0.
    const float c_signed = (p.scale_log2 == 0.f) ? 1e-30f : p.scale_log2;
    // A negative scale is applied as |c| to negated scores (s * c == (-s) * |c|), so the maximum,
    // the masks and the exponentials below have one form: the MMA warp then computes S with
    // A = -Q (the instruction descriptor's negate-A bit).
    const float c = fabsf(c_signed);
    const float tau = p.rescale_threshold;
    float m_ref = -INFINITY;  // reference max of the scaled scores (log2 units)
    float l = 0.f;            // running denominator relative to m_ref

    for (int j = 0; j < n_tiles; ++j) {
        // S_t(j), then P_t(j), in the TMEM buffer of this step (n_first: tile 0's key tiles).
        const uint32_t s_cols = tmem + lane_base + tmem_s_buf<D>(t, j, n_first);
        if (!wait_bar_warp(bar(L::hand(L::B_S_FULL, t, j, n_first)), L::hand_parity(t, j, n_first),
                           ctl, SITE_SOFTMAX_S_FULL))
            return;
        ptx::tc_fence_after();
        uint32_t sr[4][32];
        ptx::tmem_ld128(s_cols, sr);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q) ptx::reg_fence(sr[q]);

        // Keys of this tile the row may see: [k0, k0 + lim).
        const int k0 = (kv0 + j) * BN;
        const bool need_mask = (k0 + BN > p.nk) || (CAUSAL && k0 + BN - 1 > q_tile0);
        int lim = p.nk - k0;
        if constexpr (CAUSAL) lim = min(lim, row + 1 - k0);
        if (need_mask) {
            const uint32_t hidden = 0xff800000u;  // -inf
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (q * 32 + i >= lim) sr[q][i] = hidden;
        }

        // Tile maximum on the raw scores (scaling by c > 0 is monotone), as four independent
        // chains per block of 32 columns: chain c of block q covers columns c, c + 4, c + 8, ...
        // so the 3-input steps of different chains overlap.
        float mx[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float ch[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) ch[c] = __uint_as_float(sr[q][c]);
#pragma unroll
            for (int i = 4; i < 28; i += 8)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    ch[c] = ptx::fmax3(ch[c], __uint_as_float(sr[q][i + c]),
                                       __uint_as_float(sr[q][i + 4 + c]));
#pragma unroll
            for (int c = 0; c < 4; ++c)
                ch[c] = fmaxf(ch[c], __uint_as_float(sr[q][28 + c]));
            mx[q] = fmaxf(fmaxf(ch[0], ch[1]), fmaxf(ch[2], ch[3]));
        }
        const float mraw = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        const float m_tile = (mraw == INFINITY || mraw == -INFINITY) ? -INFINITY : mraw * c;

        // Lazy reference update: move m_ref only when the row max rose by more than tau.
        float corr = 1.f;
        if (m_tile > m_ref + tau || m_ref == -INFINITY) {
            const float m_new = fmaxf(m_ref, m_tile);
            corr = (m_ref == -INFINITY) ? 0.f : ptx::ex2(m_ref - m_new);
            m_ref = m_new;
        }
        const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;

        // P = 2^(s*c - m_ref), rounded to 16 bits; l sums the rounded values, so O / l is an
        // exact weighted average of V under the weights the PV product uses. P is released in two
        // halves (keys 0-63, then 64-127) so the PV product starts on the first half while the
        // second is computed.
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t pk[32];
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                const int q = 2 * h + qq;
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float x0, x1;
                    ptx::ffma2(x0, x1, __uint_as_float(sr[q][i]), __uint_as_float(sr[q][i + 1]),
                               c, neg_m);
                    // A hidden score holds -inf, so its weight is 2^-inf = 0.
                    const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                    const uint32_t u = pack2<BF16>(p0, p1);
                    ptx::add_halves<BF16>(acc[(i >> 1) & 3], acc[4 + ((i >> 1) & 3)], u);
                    pk[qq * 16 + i / 2] = u;
                }
            }
            ptx::tmem_st32(s_cols + h * 32, pk);
            if (h == 0 && j > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
                // Rescale this warp's O rows when any of them moved its reference. O_t must hold
                // every key < k0, and PV_t(j) starts only after this warp's release. With one
                // buffer per tile no wait is needed: the S_t(j) commit this warp waited on was
                // issued after PV_t(j-1). With the S ring, PV_t(j-1) may still run: wait for it.
                if constexpr (S_RING<D>) {
                    if (!wait_bar_warp(bar(L::B_O_DONE + t), (j - 1) & 1, ctl, SITE_SOFTMAX_O_DONE))
                        return;
                    ptx::tc_fence_after();
                }
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t o[32];
                    ptx::tmem_ld32(o_cols + q * 32, o);
                    ptx::tmem_wait_ld();
                    ptx::reg_fence(o);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
                    ptx::tmem_st32(o_cols + q * 32, o);
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(L::hand(h == 0 ? L::B_P_HALF : L::B_P_FULL, t, j, n_first)));
        }
        const float rowsum =
            ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        l = l * corr + rowsum;
    }
    epilogue<D, BF16>(t, tmem, sbase, p, ctl, bh, q0, split, l, m_ref, tm_o);
}

// ---------------------------------------------------------------------------------------------
// work unit of CTA b: slice bh, unit u (query rows u * 256 ...), key range split (-1: all keys).
// Causal: the longest units first, spread over all slices; otherwise the units of one slice are
// adjacent so its K/V stay hot in L2, and the units from split_begin on run as num_splits CTAs.
// ---------------------------------------------------------------------------------------------
template <bool CAUSAL>
__device__ __forceinline__ void unit_of_cta(int b, const Params& p, int& bh, int& u, int& split) {
    split = -1;
    if constexpr (CAUSAL) {
        bh = b % p.bh;
        u = p.num_units - 1 - b / p.bh;
    } else {
        int unit = b;
        if (unit >= p.split_begin) {
            const int idx = unit - p.split_begin;
            unit = p.split_begin + idx / p.num_splits;
            split = idx % p.num_splits;
        }
        u = unit % p.num_units;
        bh = unit / p.num_units;
    }
}

// ---------------------------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------------------------
template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const Params p) {
    using L = Smem<D>;
    constexpr int STAGES = L::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = ptx::smem_u32(smem);
    auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * static_cast<uint32_t>(i); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::ABORT_OFF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::TMEM_SLOT_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int wg = warp >> 2;

    // Work unit (split < 0: the whole key range, O written directly).
    int bh, u, split;
    unit_of_cta<CAUSAL>(static_cast<int>(blockIdx.x), p, bh, u, split);
    const int nkt = (p.nk + BN - 1) / BN;
    const int q0 = u * UNIT_ROWS;
    // This CTA's key tiles: [kv0, kv0 + n_tiles[t]) for query tile t.
    const int kv0 = split < 0 ? 0 : split * p.kv_tiles_per_split;
    int n_tiles[Q_TILES];
#pragma unroll
    for (int t = 0; t < Q_TILES; ++t)
        n_tiles[t] = CAUSAL ? min(nkt, (q0 + t * BM + BM - 1) / BN + 1)
                            : (split < 0 ? nkt : min(nkt - kv0, p.kv_tiles_per_split));

    const bool early = p.early_loads != 0;
    const uint32_t sq = sbase + L::Q_OFF, sk = sbase + L::K_OFF, sv = sbase + L::V_OFF;
    // TMA loads of the producer lane: Q tile t, and K tile j into its stage.
    auto load_q = [&](int t) {
        ptx::mbar_arrive_expect_tx(bar(L::B_Q_FULL + t), L::Q_TILE_BYTES);
        for (int c = 0; c < L::COL_BLOCKS; ++c)
            ptx::tma_load_3d(sq + t * L::Q_TILE_BYTES + c * (BM * 128), &tm_q, c * 64, q0 + t * BM,
                             bh, bar(L::B_Q_FULL + t));
    };
    auto load_k = [&](int j) {
        const int st = j % STAGES;
        ptx::mbar_arrive_expect_tx(bar(L::B_K_FULL + st), L::KV_BYTES);
        for (int c = 0; c < L::COL_BLOCKS; ++c)
            ptx::tma_load_3d(sk + st * L::KV_BYTES + c * (BN * 128), &tm_k, c * 64, (kv0 + j) * BN,
                             bh, bar(L::B_K_FULL + st));
    };
    if (threadIdx.x == (early ? LOAD_WARP * 32 : 0)) {
        *abort_flag = 0;
        for (int h = 0; h < L::HAND; ++h) {
            ptx::mbar_init(bar(L::B_S_FULL + h), 1);
            ptx::mbar_init(bar(L::B_P_HALF + h), BM);
            ptx::mbar_init(bar(L::B_P_FULL + h), BM);
        }
        for (int t = 0; t < Q_TILES; ++t) {
            ptx::mbar_init(bar(L::B_Q_FULL + t), 1);
            if (S_RING<D>) ptx::mbar_init(bar(L::B_O_DONE + t), 1);
            ptx::mbar_init(bar(L::B_O_READY + t), 1);
            ptx::mbar_init(bar(L::B_O_STAGED + t), 4);
            ptx::mbar_init(bar(L::B_Q_ROT + t), 8);
        }
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar(L::B_K_FULL + s), 1);
            ptx::mbar_init(bar(L::B_K_EMPTY + s), 1);
            ptx::mbar_init(bar(L::B_V_FULL + s), 1);
            ptx::mbar_init(bar(L::B_V_EMPTY + s), 1);
        }
        ptx::mbar_init(bar(L::B_DRAIN), 1);
        ptx::fence_barrier_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == LOAD_WARP && lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::prefetch_tensormap(&tm_o);
        // A first-wave CTA of a dependent launch starts while the previous kernel finishes and
        // waits for it below. Prefetching its first Q, K and V tiles into L2 first overlaps their
        // DRAM latency with that wait. The prefetch moves no data into the SM, and L2 holds the
        // one coherent copy of global memory, so it cannot make a later load see anything older
        // than what the previous kernel writes.
        if (static_cast<int>(blockIdx.x) < p.prefetch_ctas) {
            for (int c = 0; c < L::COL_BLOCKS; ++c) {
                ptx::tma_prefetch_3d(&tm_q, c * 64, q0, bh);
                ptx::tma_prefetch_3d(&tm_k, c * 64, kv0 * BN, bh);
                ptx::tma_prefetch_3d(&tm_v, c * 64, kv0 * BN, bh);
                ptx::tma_prefetch_3d(&tm_q, c * 64, q0 + BM, bh);
            }
        }
    }
    // Loads the producer lane issued before the CTA barrier (early mode): the Q tiles the first
    // products need, and K_0. Its barriers are its own, initialised above by this same thread.
    int pre_q = 0;
    bool pre_k0 = false;
    if (early && warp == LOAD_WARP && lane == 0) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        load_q(0);
        pre_q = 1;
        if (p.rope_cos != nullptr) {
            for (int t = 1; t < Q_TILES; ++t) load_q(t);
            pre_q = Q_TILES;
        }
        if (n_tiles[Q_TILES - 1] > 0) {
            load_k(0);
            pre_k0 = true;
        }
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
    // This grid is launched as a programmatic dependent of the stream's previous kernel: the set-up
    // above (shared memory, TMEM, tensor-map and L2 prefetch hints) may overlap that kernel's last
    // CTAs, and no global memory is read or written before it has completed and its writes are
    // visible (the TMA lane, in early mode, waited above before its first loads).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Likewise a grid launched after this one as a programmatic dependent (the merge of split key
    // ranges, or the next attention launch) may be scheduled once every CTA of this grid has
    // started; it waits for this grid to complete before touching global memory.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (wg == 2) {
        ptx::regs_dec<REG_MISC>();
        if (warp == LOAD_WARP) {
            // -------------------------------------------------------------- TMA producer
            if (lane == 0) {
                // Q_0, then K_0, then the other Q tiles: the first product S_0(0) needs only the
                // first two. When the kernel rotates Q, both Q tiles come first, so that their
                // rotation overlaps K_0's load. (In early mode some of these were issued before
                // the CTA barrier.)
                int q_loaded = pre_q;
                if (q_loaded == 0) {
                    load_q(0);
                    q_loaded = 1;
                }
                const bool q_first = p.rope_cos != nullptr;
                if (q_first && q_loaded < Q_TILES) {
                    for (int t = q_loaded; t < Q_TILES; ++t) load_q(t);
                    q_loaded = Q_TILES;
                }
                const int n = n_tiles[Q_TILES - 1];
                int issued = pre_k0 ? 1 : 0;
                for (int j = 0; j < n; ++j) {
                    const int st = j % STAGES;
                    const uint32_t ph = (j / STAGES) & 1;
                    if (!(j == 0 && pre_k0)) {
                        if (!wait_bar(bar(L::B_K_EMPTY + st), ph ^ 1, ctl, SITE_LOAD_K_EMPTY)) break;
                        load_k(j);
                    }
                    issued = 2 * j + 1;
                    if (j == 0 && !q_first) {
                        for (int t = 1; t < Q_TILES; ++t) load_q(t);
                        q_loaded = Q_TILES;
                    }
                    if (!wait_bar(bar(L::B_V_EMPTY + st), ph ^ 1, ctl, SITE_LOAD_V_EMPTY)) break;
                    ptx::mbar_arrive_expect_tx(bar(L::B_V_FULL + st), L::KV_BYTES);
                    for (int c = 0; c < L::COL_BLOCKS; ++c)
                        ptx::tma_load_3d(sv + st * L::KV_BYTES + c * (BN * 128), &tm_v, c * 64,
                                         (kv0 + j) * BN, bh, bar(L::B_V_FULL + st));
                    issued = 2 * j + 2;
                }
                // The CTA one wave later starts as this wave's CTAs leave. Its first tiles,
                // prefetched into L2 now that this CTA has issued all its own loads (about two
                // key steps before it ends), are there when it starts.
                const int nb = static_cast<int>(blockIdx.x) + p.next_prefetch_stride;
                if (p.next_prefetch_stride > 0 && nb < static_cast<int>(gridDim.x) && !*abort_flag) {
                    int nbh, nu, nsplit;
                    unit_of_cta<CAUSAL>(nb, p, nbh, nu, nsplit);
                    const int nkv = nsplit < 0 ? 0 : nsplit * p.kv_tiles_per_split;
                    for (int c = 0; c < L::COL_BLOCKS; ++c) {
                        ptx::tma_prefetch_3d(&tm_q, c * 64, nu * UNIT_ROWS, nbh);
                        ptx::tma_prefetch_3d(&tm_k, c * 64, nkv * BN, nbh);
                        ptx::tma_prefetch_3d(&tm_v, c * 64, nkv * BN, nbh);
                        ptx::tma_prefetch_3d(&tm_q, c * 64, nu * UNIT_ROWS + BM, nbh);
                    }
                }
                if (*abort_flag) {
                    // Drain: every copy this thread started must land before the CTA's shared
                    // memory is released. The last copy into each stage is its newest phase.
                    for (int t = 0; t < q_loaded; ++t)
                        wait_bar(bar(L::B_Q_FULL + t), 0, ctl, SITE_DRAIN, false);
                    for (int x = (issued > 2 * STAGES ? issued - 2 * STAGES : 0); x < issued; ++x) {
                        const int j = x / 2, st = j % STAGES;
                        const uint32_t ph = (j / STAGES) & 1;
                        wait_bar(bar((x & 1) ? L::B_V_FULL + st : L::B_K_FULL + st), ph, ctl,
                                 SITE_DRAIN, false);
                    }
                }
            }
            __syncwarp();
        } else if (warp == MMA_WARP) {
            // -------------------------------------------------------------- MMA issuer
            // The whole warp runs the loop (descriptors stay warp-uniform); one elected lane
            // issues the MMAs and commits.
            uint32_t leader;
            asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
                         : "=r"(leader));
            // S = Q K^T, or -(Q K^T) under a negative scale (negate-A bit of the descriptor).
            const uint32_t IDESC_S = ptx::idesc_f16(BF16, BM, BN, false, false) |
                                     (p.scale_log2 < 0.f ? ptx::IDESC_NEGATE_A : 0u);
            constexpr uint32_t IDESC_O = ptx::idesc_f16(BF16, BM, D, false, true);
            const uint32_t sq = sbase + L::Q_OFF, sk = sbase + L::K_OFF, sv = sbase + L::V_OFF;
            // S_t = Q_t K_j^T: K-dimension D in steps of 16 elements (32 bytes inside a 128-byte
            // swizzle row); Q and K tiles are K-major, 8-row swizzle atoms 1024 bytes apart, the
            // second 64 columns of D one column block further. Descriptors are built once per
            // operand tile; a step of k adds its byte offset (>> 4) to the start-address field.
            const int n0 = n_tiles[0], n1 = n_tiles[Q_TILES - 1];
            auto issue_s = [&](int t, int j) {
                const uint64_t a0 = ptx::sdesc_sw128(sq + t * L::Q_TILE_BYTES, 16, 1024);
                const uint64_t b0 = ptx::sdesc_sw128(sk + (j % STAGES) * L::KV_BYTES, 16, 1024);
                const uint32_t d = tmem + tmem_s_buf<D>(t, j, n0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk / 4) * (BM * 128) + (kk % 4) * 32) >> 4;
                    ptx::mma_ss_if(leader, d, a0 + off, b0 + off, IDESC_S, kk > 0 ? 1u : 0u);
                }
            };
            // O_t += P_t V_j over keys [64 half, 64 half + 64): P_t is the A operand from TMEM
            // (16 keys = 8 columns of 16-bit pairs); V_j is B in MN-major layout (D contiguous):
            // 16 keys = 16 rows of 128 bytes, the next 64 columns of D one column block away.
            auto issue_pv = [&](int t, int j, int half) {
                const uint64_t b0 = ptx::sdesc_sw128(sv + (j % STAGES) * L::KV_BYTES, BN * 128, 1024);
                const uint32_t a = tmem + tmem_s_buf<D>(t, j, n0);
#pragma unroll
                for (int kk = half * (BN / 32); kk < (half + 1) * (BN / 32); ++kk)
                    ptx::mma_ts_if(leader, tmem + tmem_o<D>(t), a + kk * 8,
                                   b0 + ((kk * 16 * 128) >> 4), IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
            };
            auto commit = [&](int b) { ptx::mma_commit_if(leader, bar(b)); };
            // Q_t is ready once loaded, or once rotated when the kernel applies the rotary
            // embedding to it.
            const int q_ready = p.rope_cos != nullptr ? L::B_Q_ROT : L::B_Q_FULL;
            bool ok = true;
            if constexpr (S_RING<D>) {
                // S product k (issue order of s_seq) goes to buffer k mod 3, whose previous
                // product, k - 3, has had its PV issued just before (MMAs of one thread run in
                // order, so S product k overwrites P only after that PV has read it). Tile 1
                // (n1 >= n0) is the last user of every K and V tile.
                auto seq_at = [&](int k, int& t, int& j) {
                    if (k < 2 * n0) {
                        t = k & 1;
                        j = k >> 1;
                    } else {
                        t = 1;
                        j = k - n0;
                    }
                };
                const int total = n0 + n1;
                for (int k = 0; ok && k < total + 3; ++k) {
                    if (k >= 3) {
                        int t, j;
                        seq_at(k - 3, t, j);
                        const int st = j % STAGES;
                        if (!(ok = wait_bar_warp(bar(L::B_V_FULL + st), (j / STAGES) & 1, ctl,
                                                 SITE_MMA_V_FULL) &&
                                   wait_bar_warp(bar(L::hand(L::B_P_HALF, t, j, n0)),
                                                 L::hand_parity(t, j, n0), ctl, SITE_MMA_P_FULL)))
                            break;
                        ptx::tc_fence_after();
                        issue_pv(t, j, 0);
                        if (!(ok = wait_bar_warp(bar(L::hand(L::B_P_FULL, t, j, n0)),
                                                 L::hand_parity(t, j, n0), ctl, SITE_MMA_P_FULL)))
                            break;
                        ptx::tc_fence_after();
                        issue_pv(t, j, 1);
                        commit(L::B_O_DONE + t);
                        if (j + 1 == n_tiles[t]) commit(L::B_O_READY + t);
                        if (t == Q_TILES - 1) commit(L::B_V_EMPTY + st);
                    }
                    if (k < total) {
                        int t, j;
                        seq_at(k, t, j);
                        const int st = j % STAGES;
                        if (!(ok = (j > 0 ||
                                    wait_bar_warp(bar(q_ready + t), 0, ctl, SITE_MMA_Q_FULL)) &&
                                   wait_bar_warp(bar(L::B_K_FULL + st), (j / STAGES) & 1, ctl,
                                                 SITE_MMA_K_FULL)))
                            break;
                        ptx::tc_fence_after();
                        issue_s(t, j);
                        commit(L::hand(L::B_S_FULL, t, j, n0));
                        if (t == Q_TILES - 1) commit(L::B_K_EMPTY + st);
                    }
                }
            } else {
                // Per key tile j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1). S_t(j+1) overwrites the TMEM
                // columns P_t(j) occupies, so it follows PV_t(j) (MMAs of one thread run in order).
                ok = wait_bar_warp(bar(q_ready + 0), 0, ctl, SITE_MMA_Q_FULL) &&
                     wait_bar_warp(bar(L::B_K_FULL + 0), 0, ctl, SITE_MMA_K_FULL);
                if (ok) {
                    ptx::tc_fence_after();
                    issue_s(0, 0);
                    commit(L::B_S_FULL + 0);
                    ok = wait_bar_warp(bar(q_ready + 1), 0, ctl, SITE_MMA_Q_FULL);
                }
                if (ok) {
                    ptx::tc_fence_after();
                    issue_s(1, 0);
                    commit(L::B_S_FULL + 1);
                    commit(L::B_K_EMPTY + 0);
                }
                for (int j = 0; ok && j < n1; ++j) {
                    const int st = j % STAGES, st1 = (j + 1) % STAGES;
                    const uint32_t ph1 = ((j + 1) / STAGES) & 1;
                    if (!(ok = wait_bar_warp(bar(L::B_V_FULL + st), (j / STAGES) & 1, ctl,
                                             SITE_MMA_V_FULL)))
                        break;
                    for (int t = 0; t < Q_TILES; ++t) {
                        if (j >= n_tiles[t]) continue;
                        if (!(ok = wait_bar_warp(bar(L::B_P_HALF + t), j & 1, ctl, SITE_MMA_P_FULL)))
                            break;
                        ptx::tc_fence_after();
                        issue_pv(t, j, 0);
                        if (!(ok = wait_bar_warp(bar(L::B_P_FULL + t), j & 1, ctl, SITE_MMA_P_FULL)))
                            break;
                        ptx::tc_fence_after();
                        issue_pv(t, j, 1);
                        if (j + 1 == n_tiles[t]) commit(L::B_O_READY + t);
                        if (t == Q_TILES - 1) commit(L::B_V_EMPTY + st);
                        if (j + 1 < n_tiles[t]) {
                            if (!(ok = wait_bar_warp(bar(L::B_K_FULL + st1), ph1, ctl,
                                                     SITE_MMA_K_FULL)))
                                break;
                            ptx::tc_fence_after();
                            issue_s(t, j + 1);
                            commit(L::B_S_FULL + t);
                            if (t == Q_TILES - 1) commit(L::B_K_EMPTY + st1);
                        }
                    }
                }
            }
            if (*abort_flag) {
                // Drain: wait until every MMA this warp issued has finished.
                commit(L::B_DRAIN);
                wait_bar(bar(L::B_DRAIN), 0, ctl, SITE_DRAIN, false);
            }
            __syncwarp();
        }
    } else {
        ptx::regs_inc<REG_SOFTMAX>();
        if (p.rope_cos == nullptr || rotate_q<D, BF16>(sbase, p, ctl, q0))
            softmax_role<D, BF16, CAUSAL>(wg, tmem, sbase, p, ctl, bh, q0, split, kv0, n_tiles[wg],
                                          n_tiles[0], &tm_o);
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
