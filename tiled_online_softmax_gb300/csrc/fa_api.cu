// fa_api.cu -- the C interface of libfa (declared in include/fa.h): argument checks, TMA tensor
// maps, launch of the sm_103a kernel, the device error word and the host-buffer entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <atomic>
#include <cstring>
#include <mutex>
#include <utility>

#include "fa.h"
#include "fa_fwd_kernel.cuh"
#include "fa_merge_kernel.cuh"
#include "fa_rope_kernel.cuh"
#include "fa_bwd_kernel.cuh"

namespace {

constexpr int MAX_DEVICES = 64;

thread_local char g_msg[512] = "";

fa_status fail(fa_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

fa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(FA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------------------------------------
// Kernel timer (a measurement aid, off by default): while on, every kernel launch is bracketed
// by a pair of CUDA events on its stream, so a caller can read the device time of each kernel
// kind without a profiler. Events come from a pool made when the timer starts.
// ---------------------------------------------------------------------------------------------
struct KernelTimer {
    static constexpr int MAX_PAIRS = 8192;
    std::mutex mu;
    bool on = false;
    int used = 0;
    bool overflow = false;
    cudaEvent_t ev[2 * MAX_PAIRS] = {};
    int kind[MAX_PAIRS] = {};
    int created = 0;
    double ms[FA_KERNEL_KINDS] = {};
    int launches[FA_KERNEL_KINDS] = {};
};
KernelTimer g_timer;

// Record the start event of a launch of `kind`; returns the pair index, or -1 when off.
int timer_begin(cudaStream_t s, fa_kernel_kind kind) {
    if (!__atomic_load_n(&g_timer.on, __ATOMIC_ACQUIRE)) return -1;
    std::lock_guard<std::mutex> lock(g_timer.mu);
    if (!g_timer.on) return -1;
    if (g_timer.used >= g_timer.created / 2) {
        g_timer.overflow = true;
        return -1;
    }
    const int i = g_timer.used++;
    g_timer.kind[i] = kind;
    cudaEventRecord(g_timer.ev[2 * i], s);
    return i;
}

void timer_end(cudaStream_t s, int i) {
    if (i >= 0) cudaEventRecord(g_timer.ev[2 * i + 1], s);
}

unsigned g_attr_set[MAX_DEVICES] = {};     // bit per kernel instance: smem attribute applied
std::atomic<float> g_rescale_threshold{32.0f};  // lazy-rescale threshold (log2 units)
// fp16 weights P <= 2^threshold must stay below the fp16 maximum (65504 < 2^16); bf16 has
// fp32's exponent range, and the fp32 accumulators O and l hold far larger values.
constexpr float FP16_RESCALE_THRESHOLD_MAX = 15.0f;
float rescale_threshold_for(int dtype) {
    const float t = g_rescale_threshold.load(std::memory_order_relaxed);
    return dtype == FA_F16 && t > FP16_RESCALE_THRESHOLD_MAX ? FP16_RESCALE_THRESHOLD_MAX : t;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

unsigned long long wait_timeout_ns() {
    static unsigned long long t = [] {
        const char* e = getenv("FA_WAIT_TIMEOUT_NS");
        unsigned long long v = e ? strtoull(e, nullptr, 10) : 0ull;
        return v ? v : 1000000000ull;  // 1 s
    }();
    return t;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    auto pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

fa_status validate(const void* Q, const void* K, const void* V, void* O, int64_t B, int64_t H,
                   int64_t Nq, int64_t Nk, int64_t D, float scale, int causal, int dtype,
                   bool device_ptrs) {
    if (!Q || !K || !V || !O) return fail(FA_ERR_INVALID_ARGUMENT, "null tensor pointer");
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || D < 1)
        return fail(FA_ERR_INVALID_ARGUMENT, "sizes must be >= 1 (B=%lld H=%lld Nq=%lld Nk=%lld D=%lld)",
                    (long long)B, (long long)H, (long long)Nq, (long long)Nk, (long long)D);
    if (dtype != FA_F16 && dtype != FA_BF16)
        return fail(FA_ERR_INVALID_ARGUMENT, "unknown dtype code %d", dtype);
    if (causal != 0 && causal != 1)
        return fail(FA_ERR_INVALID_ARGUMENT, "causal must be 0 or 1 (got %d)", causal);
    if (!std::isfinite(scale)) return fail(FA_ERR_INVALID_ARGUMENT, "scale is not finite");
    if (D != 64 && D != 128)
        return fail(FA_ERR_UNSUPPORTED, "head dimension %lld not supported (64 or 128)", (long long)D);
    // Limits of the launch (grid.x) and of the tensor maps (32-bit dims).
    const int64_t bh = B * H;
    if (B > (1ll << 31) || H > (1ll << 31) || bh > (1ll << 31) - 1 || Nq > (1ll << 31) - 1 ||
        Nk > (1ll << 31) - 1)
        return fail(FA_ERR_UNSUPPORTED, "problem too large for one launch");
    const int64_t units = (Nq + fa::UNIT_ROWS - 1) / fa::UNIT_ROWS;
    if (units > ((1ll << 31) - 1) / bh) return fail(FA_ERR_UNSUPPORTED, "too many tiles");
    const size_t q_bytes = size_t(bh) * size_t(Nq) * size_t(D) * 2;
    const size_t kv_bytes = size_t(bh) * size_t(Nk) * size_t(D) * 2;
    if (device_ptrs) {
        for (const void* p : {static_cast<const void*>(Q), static_cast<const void*>(K),
                              static_cast<const void*>(V), static_cast<const void*>(O)})
            if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
                return fail(FA_ERR_MISALIGNED, "tensor pointer %p is not 16-byte aligned", p);
    }
    if (overlaps(O, q_bytes, Q, q_bytes) || overlaps(O, q_bytes, K, kv_bytes) ||
        overlaps(O, q_bytes, V, kv_bytes))
        return fail(FA_ERR_INVALID_ARGUMENT, "output overlaps an input");
    return FA_OK;
}

fa_status encode_map_uncached(CUtensorMap* map, const void* base, int64_t bh, int64_t n,
                              int64_t D, int dtype) {
    auto fn = encode_fn();
    if (!fn) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(n), cuuint64_t(bh)};
    const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(n) * cuuint64_t(D) * 2};
    const cuuint32_t box[3] = {64, 128, 1};  // 128-byte rows, 128 rows (one BM or BN tile)
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map,
                    dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
    return FA_OK;
}

// Tensor maps of recent calls. A map is a pure function of (base address, slice count, rows,
// D, dtype), so a cached map stays valid whatever happened to the memory since; the cache only
// saves re-encoding for callers that reuse their buffers. Round-robin replacement.
struct MapCache {
    static constexpr int ENTRIES = 64;
    struct Entry {
        const void* base;
        int64_t bh, n, D;
        int dtype;
        bool valid;
        CUtensorMap map;
    };
    std::mutex mu;
    Entry e[ENTRIES] = {};
    int next = 0;
};
MapCache g_maps;

fa_status encode_map(CUtensorMap* map, const void* base, int64_t bh, int64_t n, int64_t D,
                     int dtype) {
    {
        std::lock_guard<std::mutex> lock(g_maps.mu);
        for (const auto& x : g_maps.e)
            if (x.valid && x.base == base && x.bh == bh && x.n == n && x.D == D && x.dtype == dtype) {
                *map = x.map;
                return FA_OK;
            }
    }
    fa_status s = encode_map_uncached(map, base, bh, n, D, dtype);
    if (s != FA_OK) return s;
    std::lock_guard<std::mutex> lock(g_maps.mu);
    auto& x = g_maps.e[g_maps.next];
    g_maps.next = (g_maps.next + 1) % MapCache::ENTRIES;
    x.base = base;
    x.bh = bh;
    x.n = n;
    x.D = D;
    x.dtype = dtype;
    x.map = *map;
    x.valid = true;
    return FA_OK;
}

std::mutex g_mutex;
int* g_err_word[MAX_DEVICES] = {};         // device error word per device (16 bytes)
int g_arch_ok[MAX_DEVICES] = {};           // 0 unknown, 1 sm_103, -1 other
int g_num_sms[MAX_DEVICES] = {};           // streaming multiprocessors of each device

// The current device, checked to be an sm_103 GPU; its SM count is read once and cached.
// Called with g_mutex held.
fa_status arch_check_locked(int* dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= MAX_DEVICES) return fail(FA_ERR_UNSUPPORTED, "device index %d", dev);
    if (g_arch_ok[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        g_num_sms[dev] = sms > 0 ? sms : 1;
        g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (g_arch_ok[dev] != 1)
        return fail(FA_ERR_UNSUPPORTED, "device %d is not an sm_103 GPU; libfa is built for sm_103a", dev);
    *dev_out = dev;
    return FA_OK;
}

// Per-device state: architecture check and the error word. Called with no lock held.
fa_status device_state(int* dev_out, int** err_out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    int dev = 0;
    fa_status s = arch_check_locked(&dev);
    if (s != FA_OK) return s;
    if (!g_err_word[dev]) {
        int* w = nullptr;
        cudaError_t e;
        if ((e = cudaMalloc(&w, 16)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(error word)");
        if ((e = cudaMemset(w, 0, 16)) != cudaSuccess) {
            cudaFree(w);
            return cuda_fail(e, "cudaMemset(error word)");
        }
        g_err_word[dev] = w;
    }
    *dev_out = dev;
    *err_out = g_err_word[dev];
    return FA_OK;
}

// Launch `kernel` as a programmatic dependent of the stream's previous kernel: its blocks may be
// scheduled while that kernel finishes, and each executes griddepcontrol.wait before it touches
// global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

template <int D, bool BF16, bool CAUSAL>
fa_status launch_instance(int dev, int inst, const CUtensorMap& mq, const CUtensorMap& mk,
                          const CUtensorMap& mv, const CUtensorMap& mo, const fa::Params& p,
                          cudaStream_t stream) {
    auto kernel = fa::fa_fwd_kernel<D, BF16, CAUSAL>;
    constexpr int smem = fa::Smem<D>::ALLOC_BYTES;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!(g_attr_set[dev] & (1u << inst))) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
            g_attr_set[dev] |= 1u << inst;
        }
    }
    const unsigned grid = static_cast<unsigned>(p.split_begin) +
                          static_cast<unsigned>(p.split_units) * static_cast<unsigned>(p.num_splits);
    const int ti = timer_begin(stream, FA_KERNEL_FWD);
    cudaError_t e = launch_pdl(kernel, grid, fa::NUM_THREADS, smem, stream, mq, mk, mv, mo, p);
    timer_end(stream, ti);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return FA_OK;
}

// Key split of a launch: units [split_begin, split_begin + split_units) run as num_splits CTAs
// each; the others run whole. The default splits nothing.
struct Split {
    int num_splits = 1;
    int kv_tiles_per_split = 0;
    int split_begin = -1;   // -1: no unit is split
    int split_units = 0;
    float* o_part = nullptr;
    float* ml_part = nullptr;
};

// Rotary embedding of Q applied inside the attention kernel (cos == nullptr: none).
struct QRope {
    const float* cos = nullptr;
    const float* sin = nullptr;
    int form = 0;
};

fa_status launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t B,
                 int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale, int causal, int dtype,
                 cudaStream_t stream, const Split& split = Split(), const QRope& rope = QRope(),
                 float* o_f32 = nullptr) {
    int dev = 0;
    int* err = nullptr;
    fa_status s = device_state(&dev, &err);
    if (s != FA_OK) return s;
    const int64_t bh = B * H;
    CUtensorMap mq, mk, mv, mo;
    if ((s = encode_map(&mq, Q, bh, Nq, D, dtype)) != FA_OK) return s;
    if ((s = encode_map(&mk, K, bh, Nk, D, dtype)) != FA_OK) return s;
    if ((s = encode_map(&mv, V, bh, Nk, D, dtype)) != FA_OK) return s;
    if ((s = encode_map(&mo, O, bh, Nq, D, dtype)) != FA_OK) return s;
    fa::Params p{};
    p.o = O;
    p.lse = LSE;
    p.err = err;
    p.bh = static_cast<int>(bh);
    p.nq = static_cast<int>(Nq);
    p.nk = static_cast<int>(Nk);
    p.num_units = static_cast<int>((Nq + fa::UNIT_ROWS - 1) / fa::UNIT_ROWS);
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.rescale_threshold = rescale_threshold_for(int(dtype));
    p.timeout_ns = wait_timeout_ns();
    const int total_units = p.num_units * p.bh;
    const bool splitting = split.split_begin >= 0 && split.split_units > 0 && split.num_splits > 1;
    p.num_splits = splitting ? split.num_splits : 1;
    p.kv_tiles_per_split = splitting ? split.kv_tiles_per_split
                                     : static_cast<int>((Nk + fa::BN - 1) / fa::BN);
    p.split_begin = splitting ? split.split_begin : total_units;
    p.split_units = splitting ? split.split_units : 0;
    p.o_part = split.o_part;
    p.ml_part = split.ml_part;
    p.rope_cos = rope.cos;
    p.rope_sin = rope.sin;
    p.rope_form = rope.form;
    p.o_f32 = o_f32;
    // Causal launches: with the first wave's tiles prefetched before the dependency wait a
    // 32-slice causal prefill takes 2.8 % less time per back-to-back launch (same binary, the
    // prefetch switched at run time); non-causal shapes, whose first wave fetches the same K and V
    // tiles many times over, took 0.5-0.8 % more (also with Q alone prefetched).
    p.prefetch_ctas = causal ? g_num_sms[dev] : 0;
    // Every CTA prefetches the first tiles of the CTA one wave later once its own loads are
    // issued: 0.8-1.0 % less time at the headline shape, 0.65 % on causal prefill (same binary
    // switched at run time, 40 rounds).
    p.next_prefetch_stride = g_num_sms[dev];
    // The TMA lane issues the first Q and K loads before the CTA-wide barrier: 0.3-1.8 % less
    // time on every workload (same binary switched at run time, 24 rounds).
    p.early_loads = 1;
    const bool bf16 = dtype == FA_BF16;
    const int inst = (D == 128 ? 4 : 0) + (bf16 ? 2 : 0) + (causal ? 1 : 0);
    switch (inst) {
        case 0: return launch_instance<64, false, false>(dev, inst, mq, mk, mv, mo, p, stream);
        case 1: return launch_instance<64, false, true>(dev, inst, mq, mk, mv, mo, p, stream);
        case 2: return launch_instance<64, true, false>(dev, inst, mq, mk, mv, mo, p, stream);
        case 3: return launch_instance<64, true, true>(dev, inst, mq, mk, mv, mo, p, stream);
        case 4: return launch_instance<128, false, false>(dev, inst, mq, mk, mv, mo, p, stream);
        case 5: return launch_instance<128, false, true>(dev, inst, mq, mk, mv, mo, p, stream);
        case 6: return launch_instance<128, true, false>(dev, inst, mq, mk, mv, mo, p, stream);
        default: return launch_instance<128, true, true>(dev, inst, mq, mk, mv, mo, p, stream);
    }
}

// Staging buffers of fa_fwd_host on each device.
struct Staging {
    void* buf = nullptr;
    size_t bytes = 0;
};
Staging g_staging[MAX_DEVICES];
// Held for the whole of an fa_fwd_host call (and by fa_release_host_buffers): calls from several
// host threads on one device run one after another over the shared staging buffer and streams.
std::mutex g_host_mu[MAX_DEVICES];

// Streams and events of fa_fwd_host's copy/compute pipeline, per device, made on first use:
// one stream copies every chunk's inputs in, back to back; two run the chunks' attention; one
// copies every chunk's output back. Per chunk, one event marks its inputs on the device and one
// its output complete, so no copy waits behind another chunk's computation or copy-out.
constexpr int HOST_PIPE_COMPUTE = 2;
constexpr int HOST_PIPE_MAX_CHUNKS = 16;
constexpr int64_t HOST_CHUNKS = 6;  // chunks of (batch, head) slices per call, at most the above
static_assert(HOST_CHUNKS <= HOST_PIPE_MAX_CHUNKS, "one pair of events per chunk");
struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaStream_t comp[HOST_PIPE_COMPUTE] = {};
    cudaEvent_t start = nullptr;
    cudaEvent_t copied[HOST_PIPE_MAX_CHUNKS] = {};
    cudaEvent_t computed[HOST_PIPE_MAX_CHUNKS] = {};
    cudaEvent_t done_in = nullptr, done_out = nullptr;
    cudaEvent_t done_comp[HOST_PIPE_COMPUTE] = {};
};
HostPipe g_host_pipe[MAX_DEVICES];

fa_status host_pipe(int dev, HostPipe** out) {
    HostPipe& hp = g_host_pipe[dev];
    if (!hp.ready) {
        cudaError_t e = cudaSuccess;
        auto stream = [&](cudaStream_t* x) {
            if (e == cudaSuccess) e = cudaStreamCreateWithFlags(x, cudaStreamNonBlocking);
        };
        auto event = [&](cudaEvent_t* x) {
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(x, cudaEventDisableTiming);
        };
        stream(&hp.in);
        stream(&hp.out);
        for (auto& x : hp.comp) stream(&x);
        event(&hp.start);
        event(&hp.done_in);
        event(&hp.done_out);
        for (auto& x : hp.done_comp) event(&x);
        for (int c = 0; c < HOST_PIPE_MAX_CHUNKS; ++c) {
            event(&hp.copied[c]);
            event(&hp.computed[c]);
        }
        if (e != cudaSuccess) return cuda_fail(e, "host pipeline streams and events");
        hp.ready = true;
    }
    *out = &hp;
    return FA_OK;
}

// ---------------------------------------------------------------------------------------------
// Allocation-free variant (fa_fwd_noalloc): the kernel's error record lives in this file-scope
// device array instead of device memory from cudaMalloc. Host code must not pass the symbol
// itself to a kernel (on the host it names a stand-in, not a device address): its device address
// comes from cudaGetSymbolAddress, once per device, with that device current.
// ---------------------------------------------------------------------------------------------
static __device__ __align__(256) int g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES / sizeof(int)];
constexpr size_t NOALLOC_RECORD_BYTES = 16;  // what the kernel needs: one error word, padded
int* g_noalloc_addr[MAX_DEVICES] = {};

fa_status noalloc_device_state(int* dev_out, int** scratch_out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    int dev = 0;
    fa_status s = arch_check_locked(&dev);
    if (s != FA_OK) return s;
    if (!g_noalloc_addr[dev]) {
        void* addr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
        g_noalloc_addr[dev] = static_cast<int*>(addr);
    }
    *dev_out = dev;
    *scratch_out = g_noalloc_addr[dev];
    return FA_OK;
}

// Effective split plan: every split gets at least one key tile.
struct SplitPlan {
    int num_splits;
    int tiles_per_split;
};

// `want` key ranges per unit (0: enough to cover `sms` SMs), clamped to [1, key tiles].
SplitPlan plan_splits(int64_t units, int64_t Nk, int64_t want, int64_t sms) {
    const int64_t nkt = (Nk + fa::BN - 1) / fa::BN;
    if (want <= 0) want = units >= sms ? 1 : (sms + units - 1) / units;  // cover the SMs
    want = want < 1 ? 1 : (want > nkt ? nkt : want);
    const int64_t per = (nkt + want - 1) / want;
    return SplitPlan{static_cast<int>((nkt + per - 1) / per), static_cast<int>(per)};
}

int64_t units_of(int64_t B, int64_t H, int64_t Nq) {
    return B * H * ((Nq + fa::UNIT_ROWS - 1) / fa::UNIT_ROWS);
}

// SM count of the current device for host-side sizing queries; `fallback` when there is no
// usable sm_103 device (such a query then describes a GPU with that many SMs).
int64_t current_sms_or(int64_t fallback) {
    std::lock_guard<std::mutex> lock(g_mutex);
    int dev = 0;
    if (arch_check_locked(&dev) != FA_OK) return fallback;
    return g_num_sms[dev];
}

// Bytes of partial state for `split_units` units split `splits` ways.
size_t workspace_bytes(int64_t split_units, int64_t Nq, int64_t D, int splits) {
    if (splits <= 1 || split_units <= 0) return 0;
    const size_t rows = size_t(split_units) * size_t(Nq < fa::UNIT_ROWS ? Nq : fa::UNIT_ROWS);
    const size_t o_bytes = (size_t(splits) * rows * size_t(D) * 4 + 255) & ~size_t(255);
    return o_bytes + size_t(splits) * rows * 8;
}

// Resident blocks per SM of the one-row merge kernel (queried once per instance).
template <int D, bool BF16>
int merge_blocks_per_sm() {
    static const int n = [] {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fa::fa_merge_kernel<D, BF16, 1, 4>,
                                                          256, 0) != cudaSuccess) {
            cudaGetLastError();
            b = 1;
        }
        return b > 0 ? b : 1;
    }();
    return n;
}

// The merge of `nrows` split rows over `ns` splits: one row a warp, unless that grid would not
// fit one wave of resident blocks on `sms` SMs and there are at most two splits; then two rows a
// warp (the same arithmetic: one group covers both splits). With more splits the two-row form
// issues its loads in more rounds, which cost more than the wave saved (11 % on a 4-split
// merge of 8192 rows). Same-box A/B of the two-row form: 1.8 % less time per step at the
// headline shape, 3.5 % on the large-magnitude workload.
template <int D, bool BF16>
cudaError_t launch_merge(cudaLaunchConfig_t cfg, int64_t sms, const float* op, const float* mp,
                         void* O, float* LSE, int64_t nrows, int ns, const fa::MergeMap& map) {
    const int64_t one_row_blocks = (nrows * 32 + 255) / 256;
    if (ns > 2 || one_row_blocks <= sms * merge_blocks_per_sm<D, BF16>()) {
        cfg.gridDim = dim3(static_cast<unsigned>(one_row_blocks));
        return cudaLaunchKernelEx(&cfg, fa::fa_merge_kernel<D, BF16, 1, 4>, op, mp, O, LSE, nrows,
                                  ns, map);
    }
    const int64_t warps = (nrows + 1) / 2;
    cfg.gridDim = dim3(static_cast<unsigned>((warps * 32 + 255) / 256));
    return cudaLaunchKernelEx(&cfg, fa::fa_merge_kernel<D, BF16, 2, 2>, op, mp, O, LSE, nrows, ns,
                              map);
}

// Launch with the units [split_begin, split_begin + split_units) split over keys, then merge
// their rows. `workspace` holds at least workspace_bytes(split_units, Nq, D, plan.num_splits).
fa_status launch_split(const void* Q, const void* K, const void* V, void* O, float* LSE,
                       int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale,
                       int dtype, cudaStream_t strm, const SplitPlan& plan, int64_t split_begin,
                       int64_t split_units, void* workspace, const QRope& rope = QRope()) {
    const int64_t split_rows = Nq < fa::UNIT_ROWS ? Nq : fa::UNIT_ROWS;
    const size_t rows = size_t(split_units) * size_t(split_rows);
    if (rows > size_t(INT32_MAX) / 32) return fail(FA_ERR_UNSUPPORTED, "too many rows to split");
    Split sp;
    sp.num_splits = plan.num_splits;
    sp.kv_tiles_per_split = plan.tiles_per_split;
    sp.split_begin = static_cast<int>(split_begin);
    sp.split_units = static_cast<int>(split_units);
    sp.o_part = static_cast<float*>(workspace);
    sp.ml_part = reinterpret_cast<float*>(
        static_cast<uint8_t*>(workspace) +
        ((size_t(plan.num_splits) * rows * size_t(D) * 4 + 255) & ~size_t(255)));
    fa_status s = launch(Q, K, V, O, LSE, B, H, Nq, Nk, D, scale, 0, dtype, strm, sp, rope);
    if (s != FA_OK) return s;
    const fa::MergeMap map{static_cast<int>(split_begin),
                           static_cast<int>((Nq + fa::UNIT_ROWS - 1) / fa::UNIT_ROWS),
                           static_cast<int>(split_rows), static_cast<int>(Nq),
                           static_cast<int>(B * H),
                           // signal the next launch early: 3.5 % less time per call on the ragged
                           // workload, 1 % on the long-context chunk (same binary, switched at
                           // run time, 30 rounds)
                           1};
    const int64_t nrows = static_cast<int64_t>(rows);
    const int64_t sms = current_sms_or(152);
    const bool bf16 = dtype == FA_BF16;
    // Programmatic dependent launch: the merge grid may be scheduled while the attention kernel's
    // last CTAs still run (they signal it at their start); each merge block first waits, in
    // griddepcontrol.wait, for the attention kernel to complete and its writes to be visible.
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = strm;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float* op = sp.o_part;
    const float* mp = sp.ml_part;
    const int ns = plan.num_splits;
    const int ti = timer_begin(strm, FA_KERNEL_MERGE);
    cudaError_t e;
    if (D == 128)
        e = bf16 ? launch_merge<128, true>(cfg, sms, op, mp, O, LSE, nrows, ns, map)
                 : launch_merge<128, false>(cfg, sms, op, mp, O, LSE, nrows, ns, map);
    else
        e = bf16 ? launch_merge<64, true>(cfg, sms, op, mp, O, LSE, nrows, ns, map)
                 : launch_merge<64, false>(cfg, sms, op, mp, O, LSE, nrows, ns, map);
    timer_end(strm, ti);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
    return FA_OK;
}

// Shortest key range worth its own CTA: each range adds the CTA's fixed cost (start-up, first
// products, epilogue: about five key steps) and a row of partial state to write and merge.
constexpr int64_t MIN_SPLIT_TILES = 2;

// Work balancing for fa_fwd / fa_fwd_lse (non-causal) on a device with `sms` SMs, by splitting
// units over keys:
//  - fewer units than half the SMs: every unit is split into floor(sms / units) key ranges of at
//    least MIN_SPLIT_TILES tiles, so that one wave covers (nearly) all SMs;
//  - a partial last wave of at most half the SMs: its units are split into 2-4 ranges, so that
//    the wave runs on (about) all SMs for a fraction of the time.
// Either way the split units times their ranges number at most `sms` CTAs, which bounds the
// partial state (balance_workspace_bytes). Returns false when nothing is worth splitting.
bool plan_balance(int64_t units, int64_t Nk, int64_t sms, SplitPlan* plan, int64_t* begin,
                  int64_t* count) {
    const int64_t nkt = (Nk + fa::BN - 1) / fa::BN;
    if (sms < 2) return false;
    if (units <= sms / 2) {
        int64_t want = sms / units;
        if (want > nkt / MIN_SPLIT_TILES) want = nkt / MIN_SPLIT_TILES;
        if (want < 2) return false;
        *plan = plan_splits(units, Nk, want, sms);
        if (plan->num_splits < 2) return false;
        *begin = 0;
        *count = units;
        return true;
    }
    const int64_t tail = units % sms;
    if (units <= sms || tail == 0 || tail > sms / 2) return false;
    int64_t want = sms / tail;
    if (want > 4) want = 4;
    if (nkt < 2 * want) return false;
    *plan = plan_splits(tail, Nk, want, sms);
    if (plan->num_splits < 2) return false;
    *begin = units - tail;
    *count = tail;
    return true;
}

// Largest partial state plan_balance can ask for on `sms` SMs: at most `sms` split CTAs, each
// with at most 256 rows of D = 128 fp32 columns and an (m, l) pair.
size_t balance_workspace_bytes(int64_t sms) {
    const size_t rows = size_t(sms) * fa::UNIT_ROWS;
    return ((rows * 128 * 4 + 255) & ~size_t(255)) + rows * 8;
}

// Workspaces of fa_fwd's key splits: per device, a pool of fixed-size slots allocated together on
// the first split call and kept until process exit (never grown or freed by a call). A call
// takes the slot its stream used last, else a slot never used, else a slot whose last use has
// finished on the GPU (its event has completed); the slot's event is recorded after the call's
// merge launch. A call that finds every slot in use by other streams' unfinished work, or whose
// stream is being captured into a CUDA graph (a graph may be replayed at any time, concurrently
// with anything), runs as one unsplit launch instead: correct, with no shared state.
constexpr int WS_SLOTS = 4;
struct WsSlot {
    void* buf = nullptr;
    cudaEvent_t done = nullptr;      // recorded after the last call's merge launch
    unsigned long long last = 0;     // id of that call's stream (unique for the process lifetime)
    bool used = false;               // `done` has been recorded at least once
    bool claimed = false;            // a host thread is launching with this slot right now
};
struct WsPool {
    bool ready = false;
    bool failed = false;
    size_t slot_bytes = 0;
    void* base = nullptr;
    WsSlot slot[WS_SLOTS];
};
WsPool g_ws_pool[MAX_DEVICES];
std::atomic<bool> g_tail_split{true};

// Set up the pool of device `dev` (g_mutex held). False if it cannot be now (that call runs
// unsplit).
bool ws_pool_ready_locked(int dev) {
    WsPool& pool = g_ws_pool[dev];
    if (pool.ready) return true;
    if (pool.failed) return false;
    const size_t bytes = balance_workspace_bytes(g_num_sms[dev]);
    void* base = nullptr;
    const cudaError_t e = cudaMalloc(&base, bytes * WS_SLOTS);
    if (e != cudaSuccess) {
        cudaGetLastError();
        // Out of memory stays out of memory: stop trying. Anything else (another thread capturing
        // a CUDA graph in global mode forbids allocation meanwhile) is retried by a later call.
        if (e == cudaErrorMemoryAllocation) pool.failed = true;
        return false;
    }
    for (int i = 0; i < WS_SLOTS; ++i) {
        if (cudaEventCreateWithFlags(&pool.slot[i].done, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            for (int j = 0; j < i; ++j) cudaEventDestroy(pool.slot[j].done);
            cudaFree(base);
            pool.failed = true;
            return false;
        }
        pool.slot[i].buf = static_cast<uint8_t*>(base) + size_t(i) * bytes;
    }
    pool.base = base;
    pool.slot_bytes = bytes;
    pool.ready = true;
    return true;
}

// Claim a slot for a split call on the stream with id `sid` (g_mutex held), or nullptr to run
// unsplit. A slot last used by the same stream needs no wait: the stream orders the calls.
WsSlot* ws_claim_locked(int dev, unsigned long long sid, size_t need) {
    if (!ws_pool_ready_locked(dev)) return nullptr;
    WsPool& pool = g_ws_pool[dev];
    if (need > pool.slot_bytes) return nullptr;
    WsSlot* pick = nullptr;
    for (WsSlot& sl : pool.slot)
        if (!pick && !sl.claimed && sl.used && sl.last == sid) pick = &sl;
    for (WsSlot& sl : pool.slot)
        if (!pick && !sl.claimed && !sl.used) pick = &sl;
    for (WsSlot& sl : pool.slot) {
        if (pick || sl.claimed) continue;
        const cudaError_t q = cudaEventQuery(sl.done);
        if (q == cudaSuccess) pick = &sl;
        else if (q != cudaErrorNotReady) cudaGetLastError();
    }
    if (pick) pick->claimed = true;
    return pick;
}

// fa_fwd / fa_fwd_lse: one launch, or some units split over keys and merged.
fa_status forward(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t B,
                  int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale, int causal,
                  int dtype, cudaStream_t strm, const QRope& rope = QRope()) {
    if (!causal && g_tail_split) {
        int dev = 0;
        int* err = nullptr;
        fa_status s = device_state(&dev, &err);
        if (s != FA_OK) return s;
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(strm, &cap);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
        SplitPlan plan;
        int64_t begin = 0, count = 0;
        WsSlot* slot = nullptr;
        unsigned long long sid = 0;
        if (cap == cudaStreamCaptureStatusNone &&
            plan_balance(units_of(B, H, Nq), Nk, g_num_sms[dev], &plan, &begin, &count)) {
            if ((e = cudaStreamGetId(strm, &sid)) != cudaSuccess) return cuda_fail(e, "cudaStreamGetId");
            std::lock_guard<std::mutex> lock(g_mutex);
            slot = ws_claim_locked(dev, sid, workspace_bytes(count, Nq, D, plan.num_splits));
        }
        if (slot) {
            s = launch_split(Q, K, V, O, LSE, B, H, Nq, Nk, D, scale, dtype, strm, plan, begin,
                             count, slot->buf, rope);
            std::lock_guard<std::mutex> lock(g_mutex);
            slot->claimed = false;
            // Recorded even after a failed launch: whatever was enqueued is covered by it.
            if ((e = cudaEventRecord(slot->done, strm)) == cudaSuccess) {
                slot->last = sid;
                slot->used = true;
            } else if (s == FA_OK) {
                return cuda_fail(e, "cudaEventRecord(workspace)");
            }
            return s;
        }
    }
    return launch(Q, K, V, O, LSE, B, H, Nq, Nk, D, scale, causal, dtype, strm, Split(), rope);
}

fa_status launch_rope(const void* X, void* Y, const float* cos_t, const float* sin_t,
                      int64_t rows_total, int64_t n, int64_t D, int form, int dtype,
                      cudaStream_t strm) {
    const int64_t work = rows_total * (D / 16);
    int64_t blocks = (work + 255) / 256;
    const int64_t max_blocks = current_sms_or(152) * 16;  // 16 blocks of 256 threads per SM
    if (blocks > max_blocks) blocks = max_blocks;
    if (blocks < 1) blocks = 1;
    auto x = static_cast<const uint16_t*>(X);
    auto y = static_cast<uint16_t*>(Y);
    const bool bf16 = dtype == FA_BF16;
    const unsigned g = static_cast<unsigned>(blocks);
    const int ti = timer_begin(strm, FA_KERNEL_ROPE);
    const int di = int(D);
    cudaError_t e;
    if (form == 0)
        e = bf16 ? launch_pdl(fa::fa_rope_kernel<true, 0>, g, 256, 0, strm, x, y, cos_t, sin_t, rows_total, n, di)
                 : launch_pdl(fa::fa_rope_kernel<false, 0>, g, 256, 0, strm, x, y, cos_t, sin_t, rows_total, n, di);
    else
        e = bf16 ? launch_pdl(fa::fa_rope_kernel<true, 1>, g, 256, 0, strm, x, y, cos_t, sin_t, rows_total, n, di)
                 : launch_pdl(fa::fa_rope_kernel<false, 1>, g, 256, 0, strm, x, y, cos_t, sin_t, rows_total, n, di);
    timer_end(strm, ti);
    if (e != cudaSuccess) return cuda_fail(e, "rope kernel launch");
    return FA_OK;
}

fa_status validate_rope(const void* X, const void* Y, const float* cos_t, const float* sin_t,
                        int64_t rows_total, int64_t n, int64_t D, int form, int dtype) {
    if (!X || !Y || !cos_t || !sin_t) return fail(FA_ERR_INVALID_ARGUMENT, "null pointer");
    if (rows_total < 1 || n < 1 || D < 1) return fail(FA_ERR_INVALID_ARGUMENT, "sizes must be >= 1");
    if (form != 0 && form != 1) return fail(FA_ERR_INVALID_ARGUMENT, "rope form must be 0 or 1");
    if (dtype != FA_F16 && dtype != FA_BF16) return fail(FA_ERR_INVALID_ARGUMENT, "unknown dtype");
    if (D % 16 != 0 || D > 512 || ((D / 16) & (D / 16 - 1)) != 0)
        return fail(FA_ERR_UNSUPPORTED, "rope needs D = 16 * 2^k, at most 512");
    for (const void* p : {X, Y, static_cast<const void*>(cos_t), static_cast<const void*>(sin_t)})
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
            return fail(FA_ERR_MISALIGNED, "rope pointer %p is not 16-byte aligned", p);
    const size_t x_bytes = size_t(rows_total) * size_t(D) * 2;
    if (X != Y && overlaps(X, x_bytes, Y, x_bytes))
        return fail(FA_ERR_INVALID_ARGUMENT, "rope output partially overlaps its input");
    return FA_OK;
}

template <int D, bool BF16, bool CAUSAL>
fa_status launch_bwd_instance(int dev, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& mv, const CUtensorMap& mdo, const fa::BwdParams& p,
                              cudaStream_t strm) {
    constexpr int smem = fa::BwdSmem<D, CAUSAL>::ALLOC_BYTES;
    constexpr int smem_q = fa::DqSmem<D>::ALLOC_BYTES;
    auto k_kv = fa::fa_bwd_dkdv_kernel<D, BF16, CAUSAL>;
    auto k_q = fa::fa_bwd_dq_kernel<D, BF16, CAUSAL>;
    static unsigned attr_set[MAX_DEVICES] = {};  // one per template instance
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!attr_set[dev]) {
            cudaError_t e;
            if ((e = cudaFuncSetAttribute(k_kv, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess ||
                (e = cudaFuncSetAttribute(k_q, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_q)) != cudaSuccess)
                return cuda_fail(e, "cudaFuncSetAttribute(backward)");
            attr_set[dev] = 1;
        }
    }
    const unsigned nkb = static_cast<unsigned>((p.nk + 127) / 128);
    const unsigned nqb = static_cast<unsigned>((p.nq + 127) / 128);
    int ti = timer_begin(strm, FA_KERNEL_BWD_DKDV);
    cudaError_t e = launch_pdl(k_kv, nkb * static_cast<unsigned>(p.bh), fa::BWD_THREADS, smem, strm,
                               mq, mk, mv, mdo, p);
    timer_end(strm, ti);
    if (e != cudaSuccess) return cuda_fail(e, "backward dK/dV launch");
    // dQ depends only on the preprocessing (complete before the dK/dV kernel started), not on
    // dK/dV: a programmatic dependent launch lets its CTAs fill the SMs the dK/dV kernel's last
    // wave leaves idle.
    ti = timer_begin(strm, FA_KERNEL_BWD_DQ);
    e = launch_pdl(k_q, nqb * static_cast<unsigned>(p.bh), fa::BWD_THREADS, smem_q, strm, mq, mk, mv, mdo, p);
    timer_end(strm, ti);
    if (e != cudaSuccess) return cuda_fail(e, "backward dQ launch");
    return FA_OK;
}

// One block of two threads: thread 0 stores at index 8 of `buf` and thread 1 at index 40, both
// checked against a stated bound of 32 elements. `buf` holds 64, so neither store can leave it;
// in the checked build the second is recorded as a violation and skipped.
__global__ void fa_bounds_selftest_kernel(int* buf) {
    const long long idx = threadIdx.x == 0 ? 8 : 40;
    if (fa::in_bounds(idx < 32, fa::BOUNDS_SELFTEST, idx)) buf[idx] = 1;
}

}  // namespace

extern "C" {

fa_status fa_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, int64_t B,
                         int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale, int causal,
                         fa_dtype dtype, void* stream) {
    fa_status s = validate(Q, K, V, O, B, H, Nq, Nk, D, scale, causal, int(dtype), true);
    if (s != FA_OK) return s;
    if (NOALLOC_RECORD_BYTES > FA_NOALLOC_SCRATCH_BYTES)
        return fail(FA_ERR_UNSUPPORTED, "request needs %zu bytes of scratch; the static array holds %d",
                    NOALLOC_RECORD_BYTES, FA_NOALLOC_SCRATCH_BYTES);
    int dev = 0;
    int* scratch = nullptr;
    if ((s = noalloc_device_state(&dev, &scratch)) != FA_OK) return s;
    auto strm = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(scratch, 0, NOALLOC_RECORD_BYTES, strm);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(scratch)");
    const int64_t bh = B * H;
    CUtensorMap mq, mk, mv, mo;
    if ((s = encode_map(&mq, Q, bh, Nq, D, int(dtype))) != FA_OK) return s;
    if ((s = encode_map(&mk, K, bh, Nk, D, int(dtype))) != FA_OK) return s;
    if ((s = encode_map(&mv, V, bh, Nk, D, int(dtype))) != FA_OK) return s;
    if ((s = encode_map(&mo, O, bh, Nq, D, int(dtype))) != FA_OK) return s;
    fa::Params p{};
    p.o = O;
    p.lse = nullptr;
    p.err = scratch;
    p.bh = static_cast<int>(bh);
    p.nq = static_cast<int>(Nq);
    p.nk = static_cast<int>(Nk);
    p.num_units = static_cast<int>((Nq + fa::UNIT_ROWS - 1) / fa::UNIT_ROWS);
    p.num_splits = 1;  // no key split: the whole computation stays in one launch
    p.kv_tiles_per_split = static_cast<int>((Nk + fa::BN - 1) / fa::BN);
    p.split_begin = p.num_units * p.bh;
    p.split_units = 0;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.rescale_threshold = rescale_threshold_for(int(dtype));
    p.timeout_ns = wait_timeout_ns();
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        p.prefetch_ctas = causal ? g_num_sms[dev] : 0;  // as in launch()
        p.next_prefetch_stride = g_num_sms[dev];
    }
    p.early_loads = 1;
    const int inst = (D == 128 ? 4 : 0) + (dtype == FA_BF16 ? 2 : 0) + (causal ? 1 : 0);
    switch (inst) {
        case 0: return launch_instance<64, false, false>(dev, inst, mq, mk, mv, mo, p, strm);
        case 1: return launch_instance<64, false, true>(dev, inst, mq, mk, mv, mo, p, strm);
        case 2: return launch_instance<64, true, false>(dev, inst, mq, mk, mv, mo, p, strm);
        case 3: return launch_instance<64, true, true>(dev, inst, mq, mk, mv, mo, p, strm);
        case 4: return launch_instance<128, false, false>(dev, inst, mq, mk, mv, mo, p, strm);
        case 5: return launch_instance<128, false, true>(dev, inst, mq, mk, mv, mo, p, strm);
        case 6: return launch_instance<128, true, false>(dev, inst, mq, mk, mv, mo, p, strm);
        default: return launch_instance<128, true, true>(dev, inst, mq, mk, mv, mo, p, strm);
    }
}

fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, int64_t B, int64_t H,
                 int64_t Nq, int64_t Nk, int64_t D, float scale, int causal, fa_dtype dtype,
                 void* stream) {
    fa_status s = validate(Q, K, V, O, B, H, Nq, Nk, D, scale, causal, int(dtype), true);
    if (s != FA_OK) return s;
    return forward(Q, K, V, O, nullptr, B, H, Nq, Nk, D, scale, causal, int(dtype),
                   static_cast<cudaStream_t>(stream));
}

fa_status fa_fwd_lse(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t B,
                     int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale, int causal,
                     fa_dtype dtype, void* stream) {
    fa_status s = validate(Q, K, V, O, B, H, Nq, Nk, D, scale, causal, int(dtype), true);
    if (s != FA_OK) return s;
    if (!LSE) return fail(FA_ERR_INVALID_ARGUMENT, "null LSE pointer");
    if (reinterpret_cast<uintptr_t>(LSE) % 4 != 0)
        return fail(FA_ERR_MISALIGNED, "LSE pointer %p is not 4-byte aligned", static_cast<void*>(LSE));
    const size_t q_bytes = size_t(B * H) * size_t(Nq) * size_t(D) * 2;
    const size_t lse_bytes = size_t(B * H) * size_t(Nq) * 4;
    const size_t kv_bytes = size_t(B * H) * size_t(Nk) * size_t(D) * 2;
    if (overlaps(LSE, lse_bytes, O, q_bytes) || overlaps(LSE, lse_bytes, Q, q_bytes) ||
        overlaps(LSE, lse_bytes, K, kv_bytes) || overlaps(LSE, lse_bytes, V, kv_bytes))
        return fail(FA_ERR_INVALID_ARGUMENT, "LSE overlaps another tensor");
    return forward(Q, K, V, O, LSE, B, H, Nq, Nk, D, scale, causal, int(dtype),
                   static_cast<cudaStream_t>(stream));
}

fa_status fa_fwd_f32out(const void* Q, const void* K, const void* V, float* O32, float* LSE,
                        int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale,
                        int causal, fa_dtype dtype, void* stream) {
    fa_status s = validate(Q, K, V, O32, B, H, Nq, Nk, D, scale, causal, int(dtype), true);
    if (s != FA_OK) return s;
    if (LSE && reinterpret_cast<uintptr_t>(LSE) % 4 != 0)
        return fail(FA_ERR_MISALIGNED, "LSE pointer is not 4-byte aligned");
    const size_t q_bytes = size_t(B * H) * size_t(Nq) * size_t(D) * 2;
    const size_t kv_bytes = size_t(B * H) * size_t(Nk) * size_t(D) * 2;
    const size_t o_bytes = size_t(B * H) * size_t(Nq) * size_t(D) * 4;
    const size_t lse_bytes = size_t(B * H) * size_t(Nq) * 4;
    if (overlaps(O32, o_bytes, Q, q_bytes) || overlaps(O32, o_bytes, K, kv_bytes) ||
        overlaps(O32, o_bytes, V, kv_bytes) || (LSE && overlaps(LSE, lse_bytes, O32, o_bytes)))
        return fail(FA_ERR_INVALID_ARGUMENT, "output overlaps another tensor");
    // The kernel's 16-bit output map is built on Q; in this mode nothing is stored through it.
    return launch(Q, K, V, const_cast<void*>(Q), LSE, B, H, Nq, Nk, D, scale, causal, int(dtype),
                  static_cast<cudaStream_t>(stream), Split(), QRope(), O32);
}

size_t fa_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D,
                                  int num_splits) {
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || D < 1) return 0;
    const int64_t units = units_of(B, H, Nq);
    return workspace_bytes(units, Nq, D,
                           plan_splits(units, Nk, num_splits, current_sms_or(152)).num_splits);
}

fa_status fa_fwd_plan(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, int causal,
                      int num_sms, fa_plan* out) {
    if (!out) return fail(FA_ERR_INVALID_ARGUMENT, "null plan pointer");
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1)
        return fail(FA_ERR_INVALID_ARGUMENT, "sizes must be >= 1");
    if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARGUMENT, "causal must be 0 or 1");
    if (D != 64 && D != 128) return fail(FA_ERR_UNSUPPORTED, "head dimension %lld not supported", (long long)D);
    if (num_sms < 0) return fail(FA_ERR_INVALID_ARGUMENT, "num_sms must be >= 0");
    int64_t sms = num_sms;
    if (sms == 0) {
        std::lock_guard<std::mutex> lock(g_mutex);
        int dev = 0;
        fa_status s = arch_check_locked(&dev);
        if (s != FA_OK) return s;
        sms = g_num_sms[dev];
    }
    const int64_t units = units_of(B, H, Nq);
    fa_plan p{};
    p.units = units;
    p.split_begin = units;
    p.num_splits = 1;
    p.tiles_per_split = static_cast<int>((Nk + fa::BN - 1) / fa::BN);
    p.ctas = units;
    p.launches = 1;
    SplitPlan plan;
    int64_t begin = 0, count = 0;
    if (!causal && g_tail_split && plan_balance(units, Nk, sms, &plan, &begin, &count)) {
        p.split_begin = begin;
        p.split_units = count;
        p.num_splits = plan.num_splits;
        p.tiles_per_split = plan.tiles_per_split;
        p.ctas = begin + count * plan.num_splits;
        p.launches = 2;
        p.workspace_bytes = workspace_bytes(count, Nq, D, plan.num_splits);
    }
    *out = p;
    return FA_OK;
}

fa_status fa_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE,
                         int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale,
                         int num_splits, fa_dtype dtype, void* workspace,
                         size_t workspace_bytes_given, void* stream) {
    fa_status s = validate(Q, K, V, O, B, H, Nq, Nk, D, scale, 0, int(dtype), true);
    if (s != FA_OK) return s;
    if (LSE && reinterpret_cast<uintptr_t>(LSE) % 4 != 0)
        return fail(FA_ERR_MISALIGNED, "LSE pointer is not 4-byte aligned");
    const int64_t units = units_of(B, H, Nq);
    const SplitPlan plan = plan_splits(units, Nk, num_splits, current_sms_or(152));
    auto strm = static_cast<cudaStream_t>(stream);
    if (plan.num_splits <= 1) return launch(Q, K, V, O, LSE, B, H, Nq, Nk, D, scale, 0, int(dtype), strm);
    const size_t need = workspace_bytes(units, Nq, D, plan.num_splits);
    if (!workspace || workspace_bytes_given < need)
        return fail(FA_ERR_INVALID_ARGUMENT, "workspace of %zu bytes needed for %d splits (got %zu)",
                    need, plan.num_splits, workspace_bytes_given);
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return fail(FA_ERR_MISALIGNED, "workspace is not 256-byte aligned");
    {
        const size_t qb = size_t(B * H) * size_t(Nq) * size_t(D) * 2;
        const size_t kb = size_t(B * H) * size_t(Nk) * size_t(D) * 2;
        if (overlaps(workspace, need, Q, qb) || overlaps(workspace, need, K, kb) ||
            overlaps(workspace, need, V, kb) || overlaps(workspace, need, O, qb) ||
            (LSE && overlaps(workspace, need, LSE, size_t(B * H) * size_t(Nq) * 4)))
            return fail(FA_ERR_INVALID_ARGUMENT, "workspace overlaps a tensor");
    }
    return launch_split(Q, K, V, O, LSE, B, H, Nq, Nk, D, scale, int(dtype), strm, plan, 0, units,
                        workspace);
}

fa_status fa_rope(const void* X, void* Y, const float* cos_t, const float* sin_t, int64_t B,
                  int64_t H, int64_t N, int64_t D, int form, fa_dtype dtype, void* stream) {
    if (B < 1 || H < 1) return fail(FA_ERR_INVALID_ARGUMENT, "sizes must be >= 1");
    fa_status s = validate_rope(X, Y, cos_t, sin_t, B * H * N, N, D, form, int(dtype));
    if (s != FA_OK) return s;
    return launch_rope(X, Y, cos_t, sin_t, B * H * N, N, D, form, int(dtype),
                       static_cast<cudaStream_t>(stream));
}

size_t fa_rope_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D) {
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || D < 1) return 0;
    return size_t(B * H) * size_t(Nk) * size_t(D) * 2;  // the rotated K
}

fa_status fa_fwd_rope(const void* Q, const void* K, const void* V, void* O, float* LSE,
                      const float* cos_q, const float* sin_q, const float* cos_k,
                      const float* sin_k, int rope_form, int64_t B, int64_t H, int64_t Nq,
                      int64_t Nk, int64_t D, float scale, int causal, fa_dtype dtype,
                      void* workspace, size_t workspace_bytes_given, void* stream) {
    fa_status s = validate(Q, K, V, O, B, H, Nq, Nk, D, scale, causal, int(dtype), true);
    if (s != FA_OK) return s;
    const size_t need = fa_rope_workspace_bytes(B, H, Nq, Nk, D);
    if (!workspace || workspace_bytes_given < need)
        return fail(FA_ERR_INVALID_ARGUMENT, "workspace of %zu bytes needed (got %zu)", need,
                    workspace_bytes_given);
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return fail(FA_ERR_MISALIGNED, "workspace is not 256-byte aligned");
    if (LSE && reinterpret_cast<uintptr_t>(LSE) % 4 != 0)
        return fail(FA_ERR_MISALIGNED, "LSE pointer is not 4-byte aligned");
    {
        const size_t qb = size_t(B * H) * size_t(Nq) * size_t(D) * 2;
        const size_t kb = size_t(B * H) * size_t(Nk) * size_t(D) * 2;
        if (overlaps(workspace, need, Q, qb) || overlaps(workspace, need, K, kb) ||
            overlaps(workspace, need, V, kb) || overlaps(workspace, need, O, qb) ||
            (LSE && overlaps(workspace, need, LSE, size_t(B * H) * size_t(Nq) * 4)))
            return fail(FA_ERR_INVALID_ARGUMENT, "workspace overlaps a tensor");
    }
    // K is rotated once by its own pass (every query block of a slice reads all of K); Q is
    // rotated inside the attention kernel, in shared memory, right after each tile's load.
    void* kr = workspace;
    if ((s = validate_rope(Q, Q, cos_q, sin_q, B * H * Nq, Nq, D, rope_form, int(dtype))) != FA_OK ||
        (s = validate_rope(K, kr, cos_k, sin_k, B * H * Nk, Nk, D, rope_form, int(dtype))) != FA_OK)
        return s;
    auto strm = static_cast<cudaStream_t>(stream);
    if ((s = launch_rope(K, kr, cos_k, sin_k, B * H * Nk, Nk, D, rope_form, int(dtype), strm)) != FA_OK)
        return s;
    QRope rope;
    rope.cos = cos_q;
    rope.sin = sin_q;
    rope.form = rope_form;
    return forward(Q, kr, V, O, LSE, B, H, Nq, Nk, D, scale, causal, int(dtype), strm, rope);
}

size_t fa_bwd_workspace_bytes(int64_t B, int64_t H, int64_t Nq) {
    if (B < 1 || H < 1 || Nq < 1) return 0;
    const size_t nq_pad = size_t((Nq + 127) / 128) * 128;
    return 2 * ((size_t(B * H) * nq_pad * 4 + 255) & ~size_t(255));
}

fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV, int64_t B, int64_t H, int64_t Nq,
                 int64_t Nk, int64_t D, float scale, int causal, fa_dtype dtype, void* workspace,
                 size_t workspace_bytes_given, void* stream) {
    fa_status s = validate(Q, K, V, dQ, B, H, Nq, Nk, D, scale, causal, int(dtype), true);
    if (s != FA_OK) return s;
    if (!O || !dO || !LSE || !dK || !dV) return fail(FA_ERR_INVALID_ARGUMENT, "null tensor pointer");
    for (const void* ptr : {O, dO, static_cast<const void*>(dK), static_cast<const void*>(dV)})
        if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
            return fail(FA_ERR_MISALIGNED, "tensor pointer %p is not 16-byte aligned", ptr);
    if (reinterpret_cast<uintptr_t>(LSE) % 4 != 0) return fail(FA_ERR_MISALIGNED, "LSE is not 4-byte aligned");
    const size_t qb = size_t(B * H) * size_t(Nq) * size_t(D) * 2, kb = size_t(B * H) * size_t(Nk) * size_t(D) * 2;
    const void* ins[] = {Q, K, V, O, dO, LSE};
    const size_t in_bytes[] = {qb, kb, kb, qb, qb, size_t(B * H) * size_t(Nq) * 4};
    const void* outs[] = {dQ, dK, dV};
    const size_t out_bytes[] = {qb, kb, kb};
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 6; ++b)
            if (overlaps(outs[a], out_bytes[a], ins[b], in_bytes[b]))
                return fail(FA_ERR_INVALID_ARGUMENT, "a gradient output overlaps an input");
        for (int b = a + 1; b < 3; ++b)
            if (overlaps(outs[a], out_bytes[a], outs[b], out_bytes[b]))
                return fail(FA_ERR_INVALID_ARGUMENT, "gradient outputs overlap");
    }
    const size_t need = fa_bwd_workspace_bytes(B, H, Nq);
    if (!workspace || workspace_bytes_given < need)
        return fail(FA_ERR_INVALID_ARGUMENT, "workspace of %zu bytes needed (got %zu)", need, workspace_bytes_given);
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return fail(FA_ERR_MISALIGNED, "workspace is not 256-byte aligned");
    for (int a = 0; a < 6; ++a)
        if (overlaps(workspace, need, ins[a], in_bytes[a]))
            return fail(FA_ERR_INVALID_ARGUMENT, "workspace overlaps an input");
    for (int a = 0; a < 3; ++a)
        if (overlaps(workspace, need, outs[a], out_bytes[a]))
            return fail(FA_ERR_INVALID_ARGUMENT, "workspace overlaps a gradient output");
    int dev = 0;
    int* err = nullptr;
    if ((s = device_state(&dev, &err)) != FA_OK) return s;
    const int64_t bh = B * H;
    const int64_t nq_pad = (Nq + 127) / 128 * 128;
    float* lse2 = static_cast<float*>(workspace);
    float* delta = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + need / 2);
    auto strm = static_cast<cudaStream_t>(stream);
    const bool bf16 = dtype == FA_BF16;
    {
        const int64_t threads = bh * nq_pad * (D / 8);
        const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
        const int ti = timer_begin(strm, FA_KERNEL_BWD_PREP);
        const int ibh = int(bh), inq = int(Nq), ipad = int(nq_pad);
        cudaError_t e;
        if (D == 128)
            e = bf16 ? launch_pdl(fa::fa_bwd_prep_kernel<128, true>, blocks, 256, 0, strm, O, dO, LSE, lse2, delta, ibh, inq, ipad)
                     : launch_pdl(fa::fa_bwd_prep_kernel<128, false>, blocks, 256, 0, strm, O, dO, LSE, lse2, delta, ibh, inq, ipad);
        else
            e = bf16 ? launch_pdl(fa::fa_bwd_prep_kernel<64, true>, blocks, 256, 0, strm, O, dO, LSE, lse2, delta, ibh, inq, ipad)
                     : launch_pdl(fa::fa_bwd_prep_kernel<64, false>, blocks, 256, 0, strm, O, dO, LSE, lse2, delta, ibh, inq, ipad);
        timer_end(strm, ti);
        if (e != cudaSuccess) return cuda_fail(e, "backward prep launch");
    }
    CUtensorMap mq, mk, mv, mdo;
    if ((s = encode_map(&mq, Q, bh, Nq, D, int(dtype))) != FA_OK ||
        (s = encode_map(&mk, K, bh, Nk, D, int(dtype))) != FA_OK ||
        (s = encode_map(&mv, V, bh, Nk, D, int(dtype))) != FA_OK ||
        (s = encode_map(&mdo, dO, bh, Nq, D, int(dtype))) != FA_OK)
        return s;
    fa::BwdParams p{};
    p.dq = dQ;
    p.dk = dK;
    p.dv = dV;
    p.lse2 = lse2;
    p.delta = delta;
    p.err = err;
    p.bh = int(bh);
    p.nq = int(Nq);
    p.nk = int(Nk);
    p.nq_pad = int(nq_pad);
    p.scale = scale;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.timeout_ns = wait_timeout_ns();
    p.next_prefetch_stride = g_num_sms[dev];
    // The load lanes issue their first blocks before the CTA-wide barrier: 0.2-0.8 % less time
    // (same binary switched at run time, 20 rounds).
    p.early_loads = 1;
    const int inst = (D == 128 ? 4 : 0) + (bf16 ? 2 : 0) + (causal ? 1 : 0);
    switch (inst) {
        case 0: return launch_bwd_instance<64, false, false>(dev, mq, mk, mv, mdo, p, strm);
        case 1: return launch_bwd_instance<64, false, true>(dev, mq, mk, mv, mdo, p, strm);
        case 2: return launch_bwd_instance<64, true, false>(dev, mq, mk, mv, mdo, p, strm);
        case 3: return launch_bwd_instance<64, true, true>(dev, mq, mk, mv, mdo, p, strm);
        case 4: return launch_bwd_instance<128, false, false>(dev, mq, mk, mv, mdo, p, strm);
        case 5: return launch_bwd_instance<128, false, true>(dev, mq, mk, mv, mdo, p, strm);
        case 6: return launch_bwd_instance<128, true, false>(dev, mq, mk, mv, mdo, p, strm);
        default: return launch_bwd_instance<128, true, true>(dev, mq, mk, mv, mdo, p, strm);
    }
}

fa_status fa_set_tail_split(int enable) {
    if (enable != 0 && enable != 1) return fail(FA_ERR_INVALID_ARGUMENT, "enable must be 0 or 1");
    g_tail_split.store(enable != 0, std::memory_order_relaxed);
    return FA_OK;
}

fa_status fa_fwd_host(const void* Q, const void* K, const void* V, void* O, int64_t B,
                      int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale, int causal,
                      fa_dtype dtype, void* stream) {
    fa_status s = validate(Q, K, V, O, B, H, Nq, Nk, D, scale, causal, int(dtype), false);
    if (s != FA_OK) return s;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= MAX_DEVICES) return fail(FA_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> host_lock(g_host_mu[dev]);
    const size_t q_bytes = size_t(B * H) * size_t(Nq) * size_t(D) * 2;
    const size_t kv_bytes = size_t(B * H) * size_t(Nk) * size_t(D) * 2;
    auto round_up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t need = 2 * round_up(q_bytes) + 2 * round_up(kv_bytes);
    Staging& st = g_staging[dev];
    if (st.bytes < need) {
        if (st.buf) cudaFree(st.buf);
        st.buf = nullptr;
        st.bytes = 0;
        if ((e = cudaMalloc(&st.buf, need)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(staging)");
        st.bytes = need;
    }
    auto* base = static_cast<uint8_t*>(st.buf);
    auto* dq = base;
    auto* dk = base + round_up(q_bytes);
    auto* dv = base + round_up(q_bytes) + round_up(kv_bytes);
    auto* dout = base + round_up(q_bytes) + 2 * round_up(kv_bytes);
    auto strm = static_cast<cudaStream_t>(stream);
    HostPipe* hp = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if ((s = host_pipe(dev, &hp)) != FA_OK) return s;
    }
    // The (batch, head) slices are independent: in chunks of slices, the inputs of every chunk
    // are copied in back to back on one stream (the link's bound), each chunk's attention runs as
    // soon as its inputs are there, and its output is copied back while later chunks' inputs are
    // still coming in (the two directions of the link work at once).
    const int64_t bh = B * H;
    const int64_t chunks = bh < HOST_CHUNKS ? bh : HOST_CHUNKS;
    const int64_t per = (bh + chunks - 1) / chunks;
    const size_t q_slice = size_t(Nq) * size_t(D) * 2, kv_slice = size_t(Nk) * size_t(D) * 2;
    auto* hq = static_cast<const uint8_t*>(Q);
    auto* hk = static_cast<const uint8_t*>(K);
    auto* hv = static_cast<const uint8_t*>(V);
    auto* ho = static_cast<uint8_t*>(O);
    if ((e = cudaEventRecord(hp->start, strm)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    // After an error part-way through, copies and launches already queued on the pipeline
    // streams would keep using the staging buffer and O: wait for them before returning.
    auto drain = [&](fa_status st) {
        cudaStreamSynchronize(hp->in);
        for (auto x : hp->comp) cudaStreamSynchronize(x);
        cudaStreamSynchronize(hp->out);
        return st;
    };
    for (cudaStream_t x : {hp->in, hp->comp[0], hp->comp[1], hp->out})
        if ((e = cudaStreamWaitEvent(x, hp->start, 0)) != cudaSuccess)
            return drain(cuda_fail(e, "cudaStreamWaitEvent"));
    for (int64_t c0 = 0, c = 0; c0 < bh; c0 += per, ++c) {
        const int64_t n = (bh - c0 < per) ? bh - c0 : per;
        const size_t qo = size_t(c0) * q_slice, ko = size_t(c0) * kv_slice;
        cudaStream_t x = hp->comp[c % HOST_PIPE_COMPUTE];
        if ((e = cudaMemcpyAsync(dq + qo, hq + qo, size_t(n) * q_slice, cudaMemcpyHostToDevice, hp->in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(dk + ko, hk + ko, size_t(n) * kv_slice, cudaMemcpyHostToDevice, hp->in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(dv + ko, hv + ko, size_t(n) * kv_slice, cudaMemcpyHostToDevice, hp->in)) != cudaSuccess ||
            (e = cudaEventRecord(hp->copied[c], hp->in)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(x, hp->copied[c], 0)) != cudaSuccess)
            return drain(cuda_fail(e, "cudaMemcpyAsync(host to device)"));
        // One launch per chunk, without the key split (chunks may run at the same time on the
        // two compute streams).
        s = launch(dq + qo, dk + ko, dv + ko, dout + qo, nullptr, 1, n, Nq, Nk, D, scale, causal,
                   int(dtype), x);
        if (s != FA_OK) return drain(s);
        if ((e = cudaEventRecord(hp->computed[c], x)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(hp->out, hp->computed[c], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(ho + qo, dout + qo, size_t(n) * q_slice, cudaMemcpyDeviceToHost, hp->out)) != cudaSuccess)
            return drain(cuda_fail(e, "cudaMemcpyAsync(device to host)"));
    }
    if ((e = cudaEventRecord(hp->done_in, hp->in)) != cudaSuccess ||
        (e = cudaEventRecord(hp->done_comp[0], hp->comp[0])) != cudaSuccess ||
        (e = cudaEventRecord(hp->done_comp[1], hp->comp[1])) != cudaSuccess ||
        (e = cudaEventRecord(hp->done_out, hp->out)) != cudaSuccess)
        return drain(cuda_fail(e, "host pipeline join"));
    for (cudaEvent_t ev : {hp->done_in, hp->done_comp[0], hp->done_comp[1], hp->done_out})
        if ((e = cudaStreamWaitEvent(strm, ev, 0)) != cudaSuccess)
            return drain(cuda_fail(e, "host pipeline join"));
    if ((e = cudaStreamSynchronize(strm)) != cudaSuccess) return drain(cuda_fail(e, "cudaStreamSynchronize"));
    return FA_OK;
}

fa_status fa_release_host_buffers(void) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= MAX_DEVICES) return FA_OK;
    std::lock_guard<std::mutex> host_lock(g_host_mu[dev]);
    if (g_staging[dev].buf) {
        e = cudaFree(g_staging[dev].buf);
        g_staging[dev] = Staging{};
        if (e != cudaSuccess) return cuda_fail(e, "cudaFree(staging)");
    }
    return FA_OK;
}

fa_status fa_timer_start(void) {
    std::lock_guard<std::mutex> lock(g_timer.mu);
    if (g_timer.on) return fail(FA_ERR_INVALID_ARGUMENT, "kernel timer already running");
    while (g_timer.created < 2 * KernelTimer::MAX_PAIRS) {
        cudaError_t e = cudaEventCreate(&g_timer.ev[g_timer.created]);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate(kernel timer)");
        ++g_timer.created;
    }
    g_timer.used = 0;
    g_timer.overflow = false;
    for (int k = 0; k < FA_KERNEL_KINDS; ++k) {
        g_timer.ms[k] = 0.0;
        g_timer.launches[k] = 0;
    }
    __atomic_store_n(&g_timer.on, true, __ATOMIC_RELEASE);
    return FA_OK;
}

fa_status fa_timer_stop(void) {
    std::lock_guard<std::mutex> lock(g_timer.mu);
    if (!g_timer.on) return fail(FA_ERR_INVALID_ARGUMENT, "kernel timer is not running");
    __atomic_store_n(&g_timer.on, false, __ATOMIC_RELEASE);
    for (int i = 0; i < g_timer.used; ++i) {
        cudaError_t e = cudaEventSynchronize(g_timer.ev[2 * i + 1]);
        float ms = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, g_timer.ev[2 * i], g_timer.ev[2 * i + 1]);
        if (e != cudaSuccess) return cuda_fail(e, "kernel timer events");
        g_timer.ms[g_timer.kind[i]] += ms;
        ++g_timer.launches[g_timer.kind[i]];
    }
    if (g_timer.overflow)
        return fail(FA_ERR_UNSUPPORTED, "more than %d launches timed; the rest were not recorded",
                    KernelTimer::MAX_PAIRS);
    return FA_OK;
}

fa_status fa_timer_read(fa_kernel_kind kind, double* total_ms, int* launches) {
    if (kind < 0 || kind >= FA_KERNEL_KINDS || !total_ms || !launches)
        return fail(FA_ERR_INVALID_ARGUMENT, "bad kernel kind or null output");
    std::lock_guard<std::mutex> lock(g_timer.mu);
    *total_ms = g_timer.ms[kind];
    *launches = g_timer.launches[kind];
    return FA_OK;
}

fa_status fa_wait_selftest(unsigned long long timeout_ns, void* stream) {
    if (timeout_ns == 0 || timeout_ns > 1000000000ull)
        return fail(FA_ERR_INVALID_ARGUMENT, "selftest timeout must be in (0, 1e9] ns");
    int dev = 0;
    int* err = nullptr;
    fa_status st = device_state(&dev, &err);
    if (st != FA_OK) return st;
    fa::fa_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, timeout_ns);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
    return FA_OK;
}

fa_status fa_wait_selftest_noalloc(unsigned long long timeout_ns, void* stream) {
    if (timeout_ns == 0 || timeout_ns > 1000000000ull)
        return fail(FA_ERR_INVALID_ARGUMENT, "selftest timeout must be in (0, 1e9] ns");
    int dev = 0;
    int* scratch = nullptr;
    fa_status st = noalloc_device_state(&dev, &scratch);
    if (st != FA_OK) return st;
    fa::fa_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(scratch, timeout_ns);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
    return FA_OK;
}

fa_status fa_last_device_error(void* stream, int* site) {
    if (site) *site = 0;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= MAX_DEVICES) return FA_OK;
    // The error word of the ordinary entry points, then the record of fa_fwd_noalloc (the static
    // array, reached through the device address looked up on that entry's first call). Reading
    // and clearing either allocates nothing.
    int* words[2];
    {
        std::lock_guard<std::mutex> lock(g_mutex);  // both are set up under this lock
        words[0] = g_err_word[dev];
        words[1] = g_noalloc_addr[dev];
    }
    int word = 0;
    for (int* w : words) {
        if (!w) continue;
        int x = 0;
        if ((e = cudaMemcpy(&x, w, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
            return cuda_fail(e, "cudaMemcpy(error word)");
        if (x == 0) continue;
        if ((e = cudaMemset(w, 0, sizeof(int))) != cudaSuccess)
            return cuda_fail(e, "cudaMemset(error word)");
        if (word == 0) word = x;
    }
    if (word == 0) return FA_OK;
    if (site) *site = word;
    if (word == fa::SITE_BWD_SMEM_LAYOUT)
        return fail(FA_ERR_UNSUPPORTED, "the dK/dV kernel could not align its shared memory (site %d)", word);
    return fail(FA_ERR_TIMEOUT, "a kernel gave up waiting at site %d", word);
}

int fa_debug_bounds_enabled(void) { return fa::kBoundsChecked ? 1 : 0; }

fa_status fa_debug_bounds_report(int* site, long long* index) {
    if (!site || !index) return fail(FA_ERR_INVALID_ARGUMENT, "null output pointer");
    *site = 0;
    *index = 0;
#ifdef FA_DEBUG_BOUNDS
    unsigned long long rec[2] = {0, 0};
    cudaError_t e = cudaMemcpyFromSymbol(rec, fa::g_bounds_record, sizeof(rec));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol(bounds record)");
    if (rec[0] != 0) {
        const unsigned long long zero[2] = {0, 0};
        if ((e = cudaMemcpyToSymbol(fa::g_bounds_record, zero, sizeof(zero))) != cudaSuccess)
            return cuda_fail(e, "cudaMemcpyToSymbol(bounds record)");
        *site = static_cast<int>(rec[0]);
        *index = static_cast<long long>(rec[1]);
    }
#endif
    return FA_OK;
}

fa_status fa_debug_bounds_selftest(int* buf, void* stream) {
    if (!fa::kBoundsChecked)
        return fail(FA_ERR_UNSUPPORTED, "this build does not check bounds (see libfa_debug.so)");
    if (!buf) return fail(FA_ERR_INVALID_ARGUMENT, "null buffer");
    if (reinterpret_cast<uintptr_t>(buf) % 4 != 0) return fail(FA_ERR_MISALIGNED, "buffer not 4-byte aligned");
    fa_bounds_selftest_kernel<<<1, 2, 0, static_cast<cudaStream_t>(stream)>>>(buf);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "bounds selftest launch");
    return FA_OK;
}

const char* fa_status_string(fa_status status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARGUMENT: return "FA_ERR_INVALID_ARGUMENT";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    }
    return "FA_ERR_UNKNOWN";
}

const char* fa_last_error_message(void) { return g_msg; }

fa_status fa_set_rescale_threshold(float log2_threshold) {
    if (!std::isfinite(log2_threshold) || log2_threshold < 0.f || log2_threshold > 64.f)
        return fail(FA_ERR_INVALID_ARGUMENT, "rescale threshold must be in [0, 64], got %g",
                    double(log2_threshold));
    g_rescale_threshold.store(log2_threshold, std::memory_order_relaxed);
    return FA_OK;
}

float fa_get_rescale_threshold(void) { return g_rescale_threshold.load(std::memory_order_relaxed); }

}  // extern "C"
