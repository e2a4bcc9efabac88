// lr_api.cu -- the C ABI declared in include/lrscan.h: argument checks, the
// per-device workspace, launch geometry, and the DEER host loop.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "lr_act.cuh"
#include "lr_launch.h"
#include "lr_tma.cuh"
#include "lrscan.h"

namespace lrs {

// cuTensorMapEncodeTiled, looked up once through the runtime (no link-time
// dependency on the driver library).
bool tma_encode(CUtensorMap* m, const void* ptr, int dtype, int64_t T, int64_t C, int box_c,
                int box_rows) {
    typedef CUresult (*encode_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static encode_fn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (encode_fn)f;
    });
    if (!fn) return false;
    const size_t es = dtype == 1 ? 2 : 4;
    const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)(C * es)};
    const cuuint32_t box[2] = {(cuuint32_t)box_c, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
              const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Retire the current epoch of a workspace (the ticket word's high half):
// ends a DEER solve, whose last launch published the next launch's
// aggregates tagged with the epoch after its own.
__global__ void k_retire_epoch(u64* tk) {
    atomicAdd(reinterpret_cast<unsigned long long*>(tk), 1ull << 32);
}

// Test hook kernel: sleeps about `ns` nanoseconds (bounded by the global
// timer), then fills x[0..n) with `value`.
__global__ void k_test_sleep_fill(float* x, int64_t n, float value, uint64_t ns) {
    if (threadIdx.x == 0) {
        uint64_t t0;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
        for (;;) {
            uint64_t t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            if (t - t0 >= ns) break;
            __nanosleep(10000);
        }
    }
    __syncthreads();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        x[i] = value;
}

// Test hook kernel: the activations the fused kernels use, elementwise.
__global__ void k_test_act(const float* __restrict__ x, float* __restrict__ th,
                           float* __restrict__ sg, float* __restrict__ em, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        th[i] = act_tanh(x[i]);
        sg[i] = act_sigmoid(x[i]);
        if (em) em[i] = act_expm1(x[i]);
    }
}

}  // namespace lrs

namespace {

using namespace lrs;

constexpr uint32_t kSpinLimit = 1u << 21;  // polls (backing off to ~1 us each): ~2 s
constexpr int kMaxIters = 4096;            // DEER kmax bound (residual slots)
// Launches counted on the host after which the packets and the ticket word
// are cleared, so that the device's epochs never wrap into packets left by
// earlier launches.
constexpr uint64_t kEpochClear = 1ull << 31;
// Workspace words: [0..1] the 64-bit ticket word (ticket counter, last retired
// epoch), [2] the sticky error bits, [3] unused, [4 ..] DEER residual slots.
constexpr int kWordErr = 2, kWordSlots = 4;
constexpr int kDeerBatch = 4;              // DEER iterations enqueued per residual read-back

thread_local char g_cuda_msg[256] = "";

int cuda_fail(cudaError_t e) {
    snprintf(g_cuda_msg, sizeof g_cuda_msg, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return LR_ERR_CUDA;
}
#define CK(x)                                  \
    do {                                       \
        cudaError_t e_ = (x);                  \
        if (e_ != cudaSuccess) return cuda_fail(e_); \
    } while (0)

// Per-device workspace.  Everything the kernels need besides the caller's
// buffers: carry packets (chunk states and aggregates), the tile ticket, the
// error word, DEER residual slots and second iterate, SRU bias partials.
struct DevWS {
    u64* pk = nullptr;           size_t pk_cap = 0;        // carry packets (state, aggregate)
    uint32_t* words = nullptr;   // ticket word, error bits, DEER residual slots (kWord*)
    float* partials = nullptr;   size_t partials_cap = 0; // floats
    void* ybuf = nullptr;        size_t ybuf_cap = 0;     // bytes
    uint32_t* host_word = nullptr;                        // pinned [kMaxIters], residual reads
    void* test_buf = nullptr;                             // timeout-test problem
    uint32_t* seq = nullptr;     size_t seq_cap = 0;      // DEER per-sequence state (words)
    unsigned long long* clamps = nullptr;                 // DEER ODE form: [kMaxIters] clamp counts
    struct DeerLast {                                     // the last solve of each DEER form
        int64_t T = -1, C = -1;
        int dtype = -1, K = 0;
    } deer_last[2];
    uint32_t* seq_host = nullptr; size_t seq_host_cap = 0;  // pinned mirror of its residuals
    uint64_t launches = 0;                                // packet launches since the last clear
    std::vector<void*> kept;                              // outgrown buffers graphs may still use
    cudaEvent_t done = nullptr;
    cudaStream_t last_stream = nullptr;
    bool has_last = false;
    int64_t bytes = 0;
};

std::mutex g_mu;
std::vector<DevWS*> g_ws;

int get_ws(DevWS** out) {
    int dev = 0;
    CK(cudaGetDevice(&dev));
    if ((int)g_ws.size() <= dev) g_ws.resize(dev + 1, nullptr);
    if (!g_ws[dev]) {
        DevWS* w = new DevWS();
        CK(cudaMalloc(&w->words, sizeof(uint32_t) * (kWordSlots + kMaxIters)));
        CK(cudaMemset(w->words, 0, sizeof(uint32_t) * (kWordSlots + kMaxIters)));
        CK(cudaHostAlloc(&w->host_word, sizeof(uint32_t) * kMaxIters, cudaHostAllocDefault));
        CK(cudaMalloc(&w->clamps, sizeof(unsigned long long) * kMaxIters));
        CK(cudaEventCreateWithFlags(&w->done, cudaEventDisableTiming));
        w->bytes = sizeof(uint32_t) * (kWordSlots + kMaxIters);
        g_ws[dev] = w;
    }
    *out = g_ws[dev];
    return LR_OK;
}

// Grow a workspace buffer to hold `need` elements.  keep: the outgrown buffer
// is kept until the process exits instead of freed -- a CUDA graph that
// captured a launch holds its address (the carry packets, the bias partials).
template <typename T>
int grow(DevWS& ws, T** p, size_t* cap, size_t need, bool zero, bool keep = false) {
    if (need <= *cap) return LR_OK;
    size_t n = need + need / 4;
    CK(cudaDeviceSynchronize());  // nothing in flight may still use the old buffer
    if (*p) {
        if (keep) {
            ws.kept.push_back(*p);
        } else {
            CK(cudaFree(*p));
            ws.bytes -= (int64_t)(*cap * sizeof(T));
        }
    }
    *p = nullptr;
    *cap = 0;
    CK(cudaMalloc((void**)p, n * sizeof(T)));
    if (zero) CK(cudaMemset(*p, 0, n * sizeof(T)));
    *cap = n;
    ws.bytes += (int64_t)(n * sizeof(T));
    return LR_OK;
}

// Order this call after the previous call on any other stream.  A call
// being captured into a CUDA graph is not ordered here: when the graph runs,
// the stream it is launched on orders it.
bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    return cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone;
}
int enter(DevWS& ws, cudaStream_t s) {
    if (capturing(s)) return LR_OK;
    if (ws.has_last && ws.last_stream != s) CK(cudaStreamWaitEvent(s, ws.done, 0));
    return LR_OK;
}
int leave(DevWS& ws, cudaStream_t s) {
    if (capturing(s)) return LR_OK;
    CK(cudaEventRecord(ws.done, s));
    ws.last_stream = s;
    ws.has_last = true;
    return LR_OK;
}
// From enter() on, every return of a call records the workspace event, the
// error returns included: work the call already enqueued is then still
// ordered before the next call on another stream.
struct Leave {
    DevWS& ws;
    cudaStream_t s;
    bool armed = true;
    Leave(DevWS& w, cudaStream_t st) : ws(w), s(st) {}
    int done() {
        armed = false;
        return leave(ws, s);
    }
    ~Leave() {
        if (armed) (void)leave(ws, s);
    }
};
u64* ticket_word(DevWS& ws) { return reinterpret_cast<u64*>(ws.words); }
// Count one launch that uses packets; clears the packets and the ticket word
// (epochs start again at 1) once every kEpochClear launches.
int count_launch(DevWS& ws, cudaStream_t s, uint64_t n = 1) {
    ws.launches += n;
    if (ws.launches < kEpochClear) return LR_OK;
    ws.launches = n;
    if (ws.pk) CK(cudaMemsetAsync(ws.pk, 0, ws.pk_cap * sizeof(u64), s));
    CK(cudaMemsetAsync(ws.words, 0, sizeof(u64), s));
    return LR_OK;
}

// Geometry + carry state for one launch of `op`.
// tma: -1 picks the TMA-staged kernels whenever they apply; 0 / 1 force the
// choice, and chain = true the chain protocol (the timeout test covers every
// kernel).
int plan(DevWS& ws, Op op, int dtype, bool vec, int64_t T, int64_t C, int64_t D, Geom* g,
         Carry* cr, cudaStream_t s, int tma = -1, bool chain = false, bool cluster = true) {
    const bool want_tma = tma < 0 ? use_tma(dtype, vec, T, C) : (tma == 1);
    const CarryPlan cp = chain ? chain_plan(op, dtype, vec, want_tma, T, C)
                               : carry_plan(op, dtype, vec, want_tma, T, C, cluster);
    const TileShape ts = cp.ts;
    g->T = T;
    g->C = C;
    g->D = D;
    set_channel_div(*g);
    g->n_chunks = cp.n_chunks;
    if ((C + ts.CW - 1) / ts.CW > INT32_MAX) return LR_ERR_TOO_LARGE;
    g->n_ct = (int)((C + ts.CW - 1) / ts.CW);
    const int64_t tiles = g->n_chunks * (int64_t)g->n_ct;
    if (tiles + cp.n_walk > INT32_MAX / 4) return LR_ERR_TOO_LARGE;
    g->n_tiles = (uint32_t)tiles;
    g->n_draws = 0;  // set by the launcher from the grid it picks
    g->ticket_base = 0;
    g->max_grid = 0;
    int st = grow(ws, &ws.pk, &ws.pk_cap, cp.inc_elems + cp.agg_elems, true, true);
    if (st) return st;
    st = count_launch(ws, s);
    if (st) return st;
    cr->inc = ws.pk;
    cr->agg = ws.pk + cp.inc_elems;
    cr->tk = ticket_word(ws);
    cr->err = ws.words + kWordErr;
    cr->epoch = 0;  // taken on the device from the ticket word
    cr->spin_limit = kSpinLimit;
    cr->mode = cp.mode;
    cr->n_walk = cp.n_walk;
    cr->wv = cp.wv;
    cr->tma = cp.tma ? 1 : 0;
    return LR_OK;
}

size_t esize(int dtype) { return dtype == LR_BF16 ? 2 : 4; }

int check_sizes(int64_t B, int64_t T, int64_t D, int dtype) {
    if (dtype != LR_F32 && dtype != LR_BF16) return LR_ERR_INVALID_ARG;
    if (B < 0 || T < 0 || D < 0) return LR_ERR_INVALID_ARG;
    const int64_t lim = (int64_t)1 << 62;
    if (B && T && D) {
        if (B > lim / T) return LR_ERR_TOO_LARGE;
        if (B * T > lim / D) return LR_ERR_TOO_LARGE;
        if (B * T * D >= lim) return LR_ERR_TOO_LARGE;
    }
    return LR_OK;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Required/optional pointer checks.  Returns status; sets *vec when every
// pointer allows the 16-byte path and D is a multiple of the vector width.
int check_ptrs(std::initializer_list<const void*> req, std::initializer_list<const void*> opt,
               std::initializer_list<const void*> params, int dtype, int64_t D, bool* vec) {
    const size_t es = esize(dtype);
    bool v = (D % kvec(dtype, true)) == 0;
    for (const void* p : req) {
        if (!p) return LR_ERR_INVALID_ARG;
        if (!aligned(p, es)) return LR_ERR_ALIGN;
        v = v && aligned(p, 16);
    }
    for (const void* p : opt) {
        if (!p) continue;
        if (!aligned(p, es)) return LR_ERR_ALIGN;
        v = v && aligned(p, 16);
    }
    for (const void* p : params) {
        if (!p) return LR_ERR_INVALID_ARG;
        if (!aligned(p, 4)) return LR_ERR_ALIGN;
        v = v && aligned(p, 16);
    }
    *vec = v;
    return LR_OK;
}

}  // namespace

#define GUARD std::lock_guard<std::mutex> lock_(g_mu)
#define TRY(x)                \
    do {                      \
        int st_ = (x);        \
        if (st_) return st_;  \
    } while (0)

extern "C" {

int lr_scan_fwd(const void* a, const void* b, const void* h0, void* h, int64_t B, int64_t T,
                int64_t D, int dtype, void* stream) {
    TRY(check_sizes(B, T, D, dtype));
    if (B * T * D == 0) return LR_OK;
    bool vec;
    TRY(check_ptrs({a, b, h}, {h0}, {}, dtype, D, &vec));
    GUARD;
    cudaStream_t s = (cudaStream_t)stream;
    DevWS* ws;
    TRY(get_ws(&ws));
    Geom g;
    Carry cr;
    TRY(enter(*ws, s));
    Leave lv(*ws, s);
    TRY(plan(*ws, OP_SCAN_FWD, dtype, vec, T, B * D, D, &g, &cr, s));
    CK(launch_scan_fwd(dtype, vec, a, b, h0, h, g, cr, s));
    return lv.done();
}

int lr_scan_bwd(const void* a, const void* h, const void* h0, const void* dh, void* da, void* db,
                void* dh0, int64_t B, int64_t T, int64_t D, int dtype, void* stream) {
    TRY(check_sizes(B, T, D, dtype));
    cudaStream_t s = (cudaStream_t)stream;
    if (B * T * D == 0) {
        if (dh0 && B * D > 0) {
            if (!aligned(dh0, esize(dtype))) return LR_ERR_ALIGN;
            CK(cudaMemsetAsync(dh0, 0, (size_t)(B * D) * esize(dtype), s));
        }
        return LR_OK;
    }
    bool vec;
    TRY(check_ptrs({a, h, dh, da, db}, {h0, dh0}, {}, dtype, D, &vec));
    GUARD;
    DevWS* ws;
    TRY(get_ws(&ws));
    Geom g;
    Carry cr;
    TRY(enter(*ws, s));
    Leave lv(*ws, s);
    TRY(plan(*ws, OP_SCAN_BWD, dtype, vec, T, B * D, D, &g, &cr, s));
    CK(launch_scan_bwd(dtype, vec, a, h, h0, dh, da, db, dh0, g, cr, s));
    return lv.done();
}

int sru_fwd(const void* xt, const void* uf, const void* ur, const void* x, const float* bf,
            const float* br, const void* c0, void* h, void* c, int64_t B, int64_t T, int64_t D,
            int dtype, void* stream) {
    TRY(check_sizes(B, T, D, dtype));
    if (B * T * D == 0) return LR_OK;
    bool vec;
    TRY(check_ptrs({xt, uf, ur, x, h, c}, {c0}, {bf, br}, dtype, D, &vec));
    GUARD;
    cudaStream_t s = (cudaStream_t)stream;
    DevWS* ws;
    TRY(get_ws(&ws));
    Geom g;
    Carry cr;
    TRY(enter(*ws, s));
    Leave lv(*ws, s);
    TRY(plan(*ws, OP_SRU_FWD, dtype, vec, T, B * D, D, &g, &cr, s));
    CK(launch_sru_fwd(dtype, vec, xt, uf, ur, x, bf, br, c0, h, c, g, cr, s));
    return lv.done();
}

int sru_bwd(const void* xt, const void* uf, const void* ur, const void* x, const float* bf,
            const float* br, const void* c0, const void* c, const void* dh, void* dxt, void* duf,
            void* dur, void* dx, float* dbf, float* dbr, void* dc0, int64_t B, int64_t T,
            int64_t D, int dtype, void* stream) {
    TRY(check_sizes(B, T, D, dtype));
    cudaStream_t s = (cudaStream_t)stream;
    if (B * T * D == 0) {
        if (D > 0) {
            if (!dbf || !dbr) return LR_ERR_INVALID_ARG;
            CK(cudaMemsetAsync(dbf, 0, (size_t)D * 4, s));
            CK(cudaMemsetAsync(dbr, 0, (size_t)D * 4, s));
        }
        if (dc0 && B * D > 0) CK(cudaMemsetAsync(dc0, 0, (size_t)(B * D) * esize(dtype), s));
        return LR_OK;
    }
    bool vec;
    TRY(check_ptrs({xt, uf, ur, x, c, dh, dxt, duf, dur, dx}, {c0, dc0}, {bf, br, dbf, dbr}, dtype,
                   D, &vec));
    GUARD;
    DevWS* ws;
    TRY(get_ws(&ws));
    Geom g;
    Carry cr;
    TRY(enter(*ws, s));
    Leave lv(*ws, s);
    TRY(plan(*ws, OP_SRU_BWD, dtype, vec, T, B * D, D, &g, &cr, s));
    TRY(grow(*ws, &ws->partials, &ws->partials_cap, (size_t)(2 * g.n_chunks * g.C + 2 * g.C), false,
             true));
    CK(launch_sru_bwd(dtype, vec, xt, uf, ur, x, bf, br, c0, c, dh, dxt, duf, dur, dx, dc0,
                      ws->partials, g, cr, s));
    CK(launch_bias_reduce(ws->partials, g.n_chunks, 2, B, D, BiasOut{{dbf, dbr}}, s));
    return lv.done();
}

int lstm_cell_fwd(const void* zf, const void* zi, const void* zc, const void* zo,
                  const float* bf, const float* bi, const float* bc, const float* bo,
                  const void* c0, void* h, void* c, int64_t B, int64_t T, int64_t D, int dtype,
                  void* stream) {
    TRY(check_sizes(B, T, D, dtype));
    if (B * T * D == 0) return LR_OK;
    bool vec;
    TRY(check_ptrs({zf, zi, zc, zo, h, c}, {c0}, {bf, bi, bc, bo}, dtype, D, &vec));
    GUARD;
    cudaStream_t s = (cudaStream_t)stream;
    DevWS* ws;
    TRY(get_ws(&ws));
    Geom g;
    Carry cr;
    TRY(enter(*ws, s));
    Leave lv(*ws, s);
    TRY(plan(*ws, OP_LSTM_FWD, dtype, vec, T, B * D, D, &g, &cr, s));
    CK(launch_lstm_fwd(dtype, vec, LstmGates{zf, zi, zc, zo}, LstmBias{bf, bi, bc, bo}, c0, h, c,
                       g, cr, s));
    return lv.done();
}

int lstm_cell_bwd(const void* zf, const void* zi, const void* zc, const void* zo,
                  const float* bf, const float* bi, const float* bc, const float* bo,
                  const void* c0, const void* c, const void* dh, void* dzf, void* dzi, void* dzc,
                  void* dzo, float* dbf, float* dbi, float* dbc, float* dbo, void* dc0, int64_t B,
                  int64_t T, int64_t D, int dtype, void* stream) {
    TRY(check_sizes(B, T, D, dtype));
    cudaStream_t s = (cudaStream_t)stream;
    if (B * T * D == 0) {
        if (D > 0) {
            for (float* db : {dbf, dbi, dbc, dbo}) {
                if (!db) return LR_ERR_INVALID_ARG;
                CK(cudaMemsetAsync(db, 0, (size_t)D * 4, s));
            }
        }
        if (dc0 && B * D > 0) CK(cudaMemsetAsync(dc0, 0, (size_t)(B * D) * esize(dtype), s));
        return LR_OK;
    }
    bool vec;
    TRY(check_ptrs({zf, zi, zc, zo, c, dh, dzf, dzi, dzc, dzo}, {c0, dc0},
                   {bf, bi, bc, bo, dbf, dbi, dbc, dbo}, dtype, D, &vec));
    GUARD;
    DevWS* ws;
    TRY(get_ws(&ws));
    Geom g;
    Carry cr;
    TRY(enter(*ws, s));
    Leave lv(*ws, s);
    TRY(plan(*ws, OP_LSTM_BWD, dtype, vec, T, B * D, D, &g, &cr, s));
    TRY(grow(*ws, &ws->partials, &ws->partials_cap, (size_t)(4 * g.n_chunks * g.C + 4 * g.C), false,
             true));
    CK(launch_lstm_bwd(dtype, vec, LstmGates{zf, zi, zc, zo}, LstmBias{bf, bi, bc, bo}, c0, c, dh,
                       LstmGates{dzf, dzi, dzc, dzo}, dc0, ws->partials, g, cr, s));
    CK(launch_bias_reduce(ws->partials, g.n_chunks, 4, B, D, BiasOut{{dbf, dbi, dbc, dbo}}, s));
    return lv.done();
}

static int grow_host(DevWS& ws, size_t need) {
    if (need <= ws.seq_host_cap) return LR_OK;
    const size_t n = need + need / 4;
    if (ws.seq_host) CK(cudaFreeHost(ws.seq_host));
    ws.seq_host = nullptr;
    ws.seq_host_cap = 0;
    CK(cudaHostAlloc(&ws.seq_host, n * sizeof(uint32_t), cudaHostAllocDefault));
    ws.seq_host_cap = n;
    return LR_OK;
}

static bool ranges_overlap(const void* a, const void* b, size_t n) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + n && y < x + n;
}

static float bits_f(uint32_t b) {
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
}

// One-pass iterations (operations with next-launch aggregates on the
// segmented walker kernel): every launch also publishes the next one's
// segment aggregates, with the next launch's epoch, into the second of two
// aggregate buffers after the packets plan() lays out, and a reduce-only pass
// before the first iteration publishes that one's: no iteration has a reduce
// pass.  onepass_begin sizes the packets
// and keeps the packet epochs from being cleared inside the solve;
// onepass_args points launch kk at its two buffers; the solve's Retire
// retires, on the device, the epoch that its last launch tagged the
// next-aggregates with, so that no later launch, of any operation, takes them
// for its own -- on every return once the first iteration was enqueued.
static int onepass_begin(DevWS& ws, Op op, int dtype, bool vec, int64_t T, int64_t C, int kmax,
                         cudaStream_t s, CarryPlan* cp, bool* on) {
    *cp = carry_plan(op, dtype, vec, use_tma(dtype, vec, T, C), T, C);
    *on = cp->mode == CARRY_WALK && cp->tma;
    if (!*on) return LR_OK;
    TRY(grow(ws, &ws.pk, &ws.pk_cap, cp->inc_elems + 2 * cp->agg_elems, true, true));
    if (ws.launches + (uint64_t)kmax + 8 >= kEpochClear) TRY(count_launch(ws, s, kEpochClear));
    return LR_OK;
}
struct Retire {
    DevWS& ws;
    cudaStream_t s;
    bool armed;
    Retire(DevWS& w, cudaStream_t st, bool on) : ws(w), s(st), armed(on) {}
    int done() {
        if (!armed) return LR_OK;
        armed = false;
        k_retire_epoch<<<1, 1, 0, s>>>(ticket_word(ws));
        CK(cudaGetLastError());
        return LR_OK;
    }
    ~Retire() { (void)done(); }
};

// The iteration count of the last solve of this DEER form (0: tanh, 1: ODE)
// and shape, 0 if none.  A solve writes iterate k to buf[(k + flip) % 2]
// (buf[1] is the caller's y) with flip chosen so that this count's iterate
// lands in y, and enqueues that many iterations before its first residual
// read-back; a wrong guess costs one copy or one more read-back, never a
// different result.
static int deer_predict(const DevWS& ws, int form, int64_t T, int64_t C, int dtype) {
    const DevWS::DeerLast& d = ws.deer_last[form];
    return d.T == T && d.C == C && d.dtype == dtype ? d.K : 0;
}
static void deer_remember(DevWS& ws, int form, int64_t T, int64_t C, int dtype, int K) {
    ws.deer_last[form] = DevWS::DeerLast{T, C, dtype, K};
}

// Launch kk >= 1 reads its aggregates from one buffer and publishes the next
// launch's into the other; launch 0 is the reduce-only pass, which publishes
// launch 1's.
static NextAgg onepass_args(DevWS& ws, const CarryPlan& cp, int kk, Carry& cr) {
    u64* agg0 = ws.pk + cp.inc_elems;  // where plan() put cr.agg
    cr.agg = (kk & 1) ? agg0 : agg0 + cp.agg_elems;
    return NextAgg{(kk & 1) ? agg0 + cp.agg_elems : agg0, 0u /* the next launch's: on the device */,
                   kk >= 1 ? 1u : 0u, kk == 0 ? 1u : 0u};
}

int deer_diag_solve_ex(const float* w, const void* u, const void* h0, const void* y_init, void* y,
                       int64_t B, int64_t T, int64_t D, float eps, int kmax, int per_sequence,
                       int* iters_out, float* resid_out, float* resid_hist, int* seq_iters,
                       float* seq_resid, int* launched_out, int dtype, void* stream) {
    TRY(check_sizes(B, T, D, dtype));
    if (!iters_out || kmax < 1 || kmax > kMaxIters || !(eps >= 0.f)) return LR_ERR_INVALID_ARG;
    if (per_sequence != 0 && per_sequence != 1) return LR_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (launched_out) *launched_out = 0;
    if (B * T * D == 0) {
        *iters_out = 0;
        if (resid_out) *resid_out = 0.f;
        for (int64_t b = 0; b < B; ++b) {
            if (seq_iters) seq_iters[b] = 0;
            if (seq_resid) seq_resid[b] = 0.f;
        }
        return LR_OK;
    }
    bool vec;
    TRY(check_ptrs({u, y}, {h0, y_init}, {w}, dtype, D, &vec));
    const size_t nbytes = (size_t)(B * T * D) * esize(dtype);
    if (y_init && y_init != y && ranges_overlap(y_init, y, nbytes)) return LR_ERR_INVALID_ARG;
    GUARD;
    DevWS* ws;
    TRY(get_ws(&ws));
    {
        size_t cap = ws->ybuf_cap;
        char* p = (char*)ws->ybuf;
        TRY(grow(*ws, &p, &cap, nbytes, false));
        ws->ybuf = p;
        ws->ybuf_cap = cap;
    }
    // per-sequence state: [kmax][B] residual slots, [B] stop flags, [B]
    // iteration counts, the all-done word
    uint32_t *sq_slots = nullptr, *sq_done = nullptr, *sq_all = nullptr;
    int32_t* sq_iters = nullptr;
    const size_t sq_words = (size_t)kmax * (size_t)B + 2 * (size_t)B + 1;
    if (per_sequence) {
        TRY(grow(*ws, &ws->seq, &ws->seq_cap, sq_words, false));
        // pinned mirror: the residual slots, the all-done word, the counts
        TRY(grow_host(*ws, (size_t)kmax * (size_t)B + 1 + (size_t)B));
        sq_slots = ws->seq;
        sq_done = sq_slots + (size_t)kmax * B;
        sq_iters = reinterpret_cast<int32_t*>(sq_done + B);
        sq_all = reinterpret_cast<uint32_t*>(sq_iters + B);
    }
    TRY(enter(*ws, s));
    Leave lv(*ws, s);
    CarryPlan cp;
    bool onepass;
    TRY(onepass_begin(*ws, OP_DEER, dtype, vec, T, B * D, kmax, s, &cp, &onepass));
    Retire rt(*ws, s, onepass);
    if (per_sequence) CK(cudaMemsetAsync(ws->seq, 0, sq_words * sizeof(uint32_t), s));
    uint32_t* slots = ws->words + kWordSlots;
    CK(cudaMemsetAsync(slots, 0, sizeof(uint32_t) * kmax, s));
    // iterate k writes buf[(k + flip) % 2]; buf[1] is the caller's y.
    // Iteration 1 reads the initial guess (a guess passed in y itself is first
    // copied to buf[0], and then iteration 1 writes y: flip = 0).  The first
    // batch is the last solve's iteration count (deer_predict), later ones
    // kDeerBatch, with one residual read-back per batch; an iteration enqueued
    // after the solve stopped returns at once (it sees its predecessor's
    // residual, or the all-done word, on the device).
    void* buf[2] = {ws->ybuf, y};
    const void* y0 = y_init;
    const bool in_place = y_init != nullptr && y_init == y;
    if (in_place) {
        CK(cudaMemcpyAsync(ws->ybuf, y_init, nbytes, cudaMemcpyDeviceToDevice, s));
        y0 = ws->ybuf;
    }
    const int kp = per_sequence ? 0 : deer_predict(*ws, 0, T, B * D, dtype);
    const int flip = kp > 0 && !in_place ? (kp + 1) & 1 : 0;
    auto tgt = [&](int kk) { return buf[(kk + flip) & 1]; };
    int k = 0, status = LR_ERR_NOT_CONVERGED;
    float rho = 0.f;
    int launched = 0;
    int kernels = 0;  // every kernel the solve enqueues
    bool done = false;
    if (onepass) {  // iteration 1's segment aggregates, from the initial guess
        Geom g;
        Carry cr;
        TRY(plan(*ws, OP_DEER, dtype, vec, T, B * D, D, &g, &cr, s));
        const NextAgg nx = onepass_args(*ws, cp, 0, cr);
        CK(launch_deer_iter(dtype, vec, w, u, h0, y0, tgt(1), slots, nullptr, eps, nx,
                            DeerSeq{nullptr, nullptr, nullptr}, g, cr, s));
        ++kernels;
    }
    while (!done && launched < kmax) {
        const int first = launched;
        const int want = first == 0 && kp > 0 ? kp : kDeerBatch;
        const int nb = kmax - launched < want ? kmax - launched : want;
        for (int i = 0; i < nb; ++i) {
            const int kk = ++launched;
            Geom g;
            Carry cr;
            TRY(plan(*ws, OP_DEER, dtype, vec, T, B * D, D, &g, &cr, s));
            const NextAgg nx = onepass ? onepass_args(*ws, cp, kk, cr) : NextAgg{nullptr, 0u, 0u, 0u};
            DeerSeq sq{nullptr, nullptr, nullptr};
            if (per_sequence) sq = DeerSeq{sq_slots + (size_t)(kk - 1) * B, sq_done, sq_all};
            CK(launch_deer_iter(dtype, vec, w, u, h0, kk == 1 ? y0 : tgt(kk - 1), tgt(kk),
                                slots + (kk - 1),
                                kk == 1 || per_sequence ? nullptr : slots + (kk - 2), eps, nx, sq, g,
                                cr, s));
            ++kernels;
            if (per_sequence) {
                CK(launch_deer_seq_update(sq_slots + (size_t)(kk - 1) * B, sq_done, sq_iters, sq_all,
                                          B, eps, kk, s));
                ++kernels;
            }
        }
        if (!per_sequence) {
            CK(cudaMemcpyAsync(ws->host_word + first, slots + first, sizeof(uint32_t) * nb,
                               cudaMemcpyDeviceToHost, s));
            CK(cudaStreamSynchronize(s));
            for (k = first + 1; k <= launched; ++k) {
                rho = bits_f(ws->host_word[k - 1]);
                if (resid_hist) resid_hist[k - 1] = rho;
                if (!(rho <= 3.4e38f)) { status = LR_ERR_NONFINITE; done = true; break; }
                if (rho < eps) { status = LR_OK; done = true; break; }
            }
        } else {
            uint32_t* hs = ws->seq_host;
            CK(cudaMemcpyAsync(hs + (size_t)first * B, sq_slots + (size_t)first * B,
                               sizeof(uint32_t) * (size_t)nb * B, cudaMemcpyDeviceToHost, s));
            CK(cudaMemcpyAsync(hs + (size_t)kmax * B, sq_all, sizeof(uint32_t),
                               cudaMemcpyDeviceToHost, s));
            CK(cudaStreamSynchronize(s));
            for (int kk = first + 1; kk <= launched; ++kk) {  // max over the sequences still running
                uint32_t m = 0;
                for (int64_t b = 0; b < B; ++b) m = hs[(size_t)(kk - 1) * B + b] > m ? hs[(size_t)(kk - 1) * B + b] : m;
                if (resid_hist) resid_hist[kk - 1] = bits_f(m);
            }
            done = hs[(size_t)kmax * B] != 0;
        }
    }
    if (onepass) ++kernels;  // the epoch retire below
    TRY(rt.done());
    if (!per_sequence) {
        if (k > kmax) k = kmax;
        if (tgt(k) != y) CK(cudaMemcpyAsync(y, ws->ybuf, nbytes, cudaMemcpyDeviceToDevice, s));
        if (status != LR_ERR_NONFINITE) deer_remember(*ws, 0, T, B * D, dtype, k);
        *iters_out = k;
        if (resid_out) *resid_out = rho;
        for (int64_t b = 0; b < B; ++b) {
            if (seq_iters) seq_iters[b] = k;
            if (seq_resid) seq_resid[b] = rho;
        }
    } else {
        // every sequence's last iterate into y; counts and final residuals
        CK(launch_deer_seq_gather(ws->ybuf, y, sq_iters, launched, T, B * D, D, dtype, s));
        ++kernels;
        int32_t* hi = reinterpret_cast<int32_t*>(ws->seq_host + (size_t)kmax * B + 1);
        CK(cudaMemcpyAsync(hi, sq_iters, sizeof(int32_t) * (size_t)B, cudaMemcpyDeviceToHost, s));
        CK(cudaStreamSynchronize(s));
        int kmx = 0;
        float rmx = 0.f;
        bool nonfinite = false, open = false;
        for (int64_t b = 0; b < B; ++b) {
            const int kb = hi[b] > 0 ? hi[b] : launched;  // never stopped: ran every iteration
            const float rb = bits_f(ws->seq_host[(size_t)(kb - 1) * B + b]);
            if (!(rb <= 3.4e38f)) nonfinite = true;
            else if (!(rb < eps)) open = true;
            if (seq_iters) seq_iters[b] = kb;
            if (seq_resid) seq_resid[b] = rb;
            kmx = kb > kmx ? kb : kmx;
            rmx = rb > rmx || !(rb <= 3.4e38f) ? rb : rmx;
        }
        status = nonfinite ? LR_ERR_NONFINITE : open ? LR_ERR_NOT_CONVERGED : LR_OK;
        *iters_out = kmx;
        if (resid_out) *resid_out = rmx;
    }
    if (launched_out) *launched_out = kernels;
    TRY(lv.done());
    return status;
}

int deer_diag_solve(const float* w, const void* u, const void* h0, void* y, int64_t B, int64_t T,
                    int64_t D, float eps, int kmax, int* iters_out, float* resid_out,
                    float* resid_hist, int dtype, void* stream) {
    return deer_diag_solve_ex(w, u, h0, nullptr, y, B, T, D, eps, kmax, 0, iters_out, resid_out,
                              resid_hist, nullptr, nullptr, nullptr, dtype, stream);
}

int deer_ode_solve(const float* w, const void* u, const float* dt, const void* h0, void* y,
                   int64_t B, int64_t T, int64_t D, float eps, int kmax, int* iters_out,
                   float* resid_out, float* resid_hist, int64_t* clamps_out, int dtype,
                   void* stream) {
    TRY(check_sizes(B, T, D, dtype));
    if (!iters_out || kmax < 1 || kmax > kMaxIters || !(eps >= 0.f)) return LR_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (B * T * D == 0) {
        *iters_out = 0;
        if (resid_out) *resid_out = 0.f;
        if (clamps_out) *clamps_out = 0;
        return LR_OK;
    }
    bool vec;
    TRY(check_ptrs({u, y}, {h0}, {w, dt}, dtype, D, &vec));
    GUARD;
    DevWS* ws;
    TRY(get_ws(&ws));
    const size_t nbytes = (size_t)(B * T * D) * esize(dtype);
    {
        size_t cap = ws->ybuf_cap;
        char* p = (char*)ws->ybuf;
        TRY(grow(*ws, &p, &cap, nbytes, false));
        ws->ybuf = p;
        ws->ybuf_cap = cap;
    }
    TRY(enter(*ws, s));
    Leave lv(*ws, s);
    CarryPlan cp;
    bool onepass;
    TRY(onepass_begin(*ws, OP_DEER_ODE, dtype, vec, T, B * D, kmax, s, &cp, &onepass));
    Retire rt(*ws, s, onepass);
    uint32_t* slots = ws->words + kWordSlots;
    CK(cudaMemsetAsync(slots, 0, sizeof(uint32_t) * kmax, s));
    CK(cudaMemsetAsync(ws->clamps, 0, sizeof(unsigned long long) * kmax, s));
    // as deer_diag_solve_ex: iterate k writes buf[(k + flip) % 2] (buf[1] is
    // y), the first batch is the last solve's count, later ones kDeerBatch
    void* buf[2] = {ws->ybuf, y};
    const int kp = deer_predict(*ws, 1, T, B * D, dtype);
    const int flip = kp > 0 ? (kp + 1) & 1 : 0;
    auto tgt = [&](int kk) { return buf[(kk + flip) & 1]; };
    int k = 0, status = LR_ERR_NOT_CONVERGED;
    float rho = 0.f;
    int launched = 0;
    bool done = false;
    if (onepass) {  // iteration 1's segment aggregates, from the zero guess
        Geom g;
        Carry cr;
        TRY(plan(*ws, OP_DEER_ODE, dtype, vec, T, B * D, D, &g, &cr, s));
        const NextAgg nx = onepass_args(*ws, cp, 0, cr);
        CK(launch_deer_ode_iter(dtype, vec, w, u, dt, h0, nullptr, tgt(1), slots, nullptr, eps,
                                ws->clamps, nx, g, cr, s));
    }
    while (!done && launched < kmax) {
        const int first = launched;
        const int want = first == 0 && kp > 0 ? kp : kDeerBatch;
        const int nb = kmax - launched < want ? kmax - launched : want;
        for (int i = 0; i < nb; ++i) {
            const int kk = ++launched;
            Geom g;
            Carry cr;
            TRY(plan(*ws, OP_DEER_ODE, dtype, vec, T, B * D, D, &g, &cr, s));
            const NextAgg nx = onepass ? onepass_args(*ws, cp, kk, cr) : NextAgg{nullptr, 0u, 0u, 0u};
            CK(launch_deer_ode_iter(dtype, vec, w, u, dt, h0, kk == 1 ? nullptr : tgt(kk - 1), tgt(kk),
                                    slots + (kk - 1),
                                    kk == 1 ? nullptr : slots + (kk - 2), eps,
                                    ws->clamps + (kk - 1), nx, g, cr, s));
        }
        CK(cudaMemcpyAsync(ws->host_word + first, slots + first, sizeof(uint32_t) * nb,
                           cudaMemcpyDeviceToHost, s));
        CK(cudaStreamSynchronize(s));
        for (k = first + 1; k <= launched; ++k) {
            rho = bits_f(ws->host_word[k - 1]);
            if (resid_hist) resid_hist[k - 1] = rho;
            if (!(rho <= 3.4e38f)) { status = LR_ERR_NONFINITE; done = true; break; }
            if (rho < eps) { status = LR_OK; done = true; break; }
        }
    }
    TRY(rt.done());
    if (k > kmax) k = kmax;
    if (tgt(k) != y) CK(cudaMemcpyAsync(y, ws->ybuf, nbytes, cudaMemcpyDeviceToDevice, s));
    if (status != LR_ERR_NONFINITE) deer_remember(*ws, 1, T, B * D, dtype, k);
    if (clamps_out) {
        unsigned long long n = 0;
        CK(cudaMemcpyAsync(&n, ws->clamps + (k - 1), sizeof n, cudaMemcpyDeviceToHost, s));
        CK(cudaStreamSynchronize(s));
        *clamps_out = (int64_t)n;
    }
    *iters_out = k;
    if (resid_out) *resid_out = rho;
    TRY(lv.done());
    return status;
}

int deer_diag_bwd(const float* w, const void* y, const void* h0, const void* dy, void* du,
                  float* dw, void* dh0, int64_t B, int64_t T, int64_t D, int dtype, void* stream) {
    TRY(check_sizes(B, T, D, dtype));
    cudaStream_t s = (cudaStream_t)stream;
    if (B * T * D == 0) {
        if (D > 0) {
            if (!dw) return LR_ERR_INVALID_ARG;
            CK(cudaMemsetAsync(dw, 0, (size_t)D * 4, s));
        }
        if (dh0 && B * D > 0) CK(cudaMemsetAsync(dh0, 0, (size_t)(B * D) * esize(dtype), s));
        return LR_OK;
    }
    bool vec;
    TRY(check_ptrs({y, dy, du}, {h0, dh0}, {w, dw}, dtype, D, &vec));
    GUARD;
    DevWS* ws;
    TRY(get_ws(&ws));
    Geom g;
    Carry cr;
    TRY(enter(*ws, s));
    Leave lv(*ws, s);
    TRY(plan(*ws, OP_DEER_BWD, dtype, vec, T, B * D, D, &g, &cr, s));
    TRY(grow(*ws, &ws->partials, &ws->partials_cap, (size_t)(g.n_chunks * g.C + g.C), false, true));
    CK(launch_deer_bwd(dtype, vec, w, y, h0, dy, du, dh0, ws->partials, g, cr, s));
    CK(launch_bias_reduce(ws->partials, g.n_chunks, 1, B, D, BiasOut{{dw}}, s));
    return lv.done();
}

int lr_last_error(void) {
    GUARD;
    DevWS* ws;
    TRY(get_ws(&ws));
    CK(cudaDeviceSynchronize());
    uint32_t bits = 0;
    CK(cudaMemcpy(&bits, ws->words + kWordErr, sizeof bits, cudaMemcpyDeviceToHost));
    CK(cudaMemset(ws->words + kWordErr, 0, sizeof(uint32_t)));
    // a launch that gave up may have stopped drawing tickets before the
    // drawer that resets the counter: reset it here (nothing is in flight),
    // and retire its epoch
    if (bits) {
        u64 tw = 0;
        CK(cudaMemcpy(&tw, ws->words, sizeof tw, cudaMemcpyDeviceToHost));
        tw = (u64)epoch_after((uint32_t)(tw >> 32)) << 32;
        CK(cudaMemcpy(ws->words, &tw, sizeof tw, cudaMemcpyHostToDevice));
    }
    if (bits & ERRBIT_TIMEOUT) return LR_ERR_TIMEOUT;
    return LR_OK;
}

const char* lr_status_str(int st) {
    switch (st) {
        case LR_OK: return "ok";
        case LR_ERR_INVALID_ARG: return "invalid argument";
        case LR_ERR_ALIGN: return "pointer not aligned to its element size";
        case LR_ERR_CUDA: return "CUDA runtime error";
        case LR_ERR_TIMEOUT: return "a carry wait ran out on the device";
        case LR_ERR_NONFINITE: return "non-finite residual";
        case LR_ERR_NOT_CONVERGED: return "not converged within kmax iterations";
        case LR_ERR_TOO_LARGE: return "problem size beyond the supported range";
        default: return "unknown status";
    }
}

const char* lr_cuda_error_string(void) { return g_cuda_msg; }

int64_t lr_workspace_bytes(void) {
    GUARD;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if ((int)g_ws.size() <= dev || !g_ws[dev]) return 0;
    return g_ws[dev]->bytes;
}

static_assert((int)LR_OP_SCAN_FWD == (int)OP_SCAN_FWD && (int)LR_OP_SCAN_BWD == (int)OP_SCAN_BWD &&
                  (int)LR_OP_SRU_FWD == (int)OP_SRU_FWD && (int)LR_OP_SRU_BWD == (int)OP_SRU_BWD &&
                  (int)LR_OP_DEER == (int)OP_DEER && (int)LR_OP_DEER_BWD == (int)OP_DEER_BWD &&
                  (int)LR_OP_LSTM_FWD == (int)OP_LSTM_FWD && (int)LR_OP_LSTM_BWD == (int)OP_LSTM_BWD &&
                  (int)LR_OP_DEER_ODE == (int)OP_DEER_ODE && (int)OP_DEER_ODE + 1 == (int)OP_COUNT,
              "lr_op follows the library's operation order");
static_assert(LR_PROTO_CHAIN == CARRY_CHAIN && LR_PROTO_WALK == CARRY_WALK &&
                  LR_PROTO_LOOK == CARRY_LOOK && LR_PROTO_CLUSTER == CARRY_CLUSTER,
              "lr_protocol follows the carry modes");

int lr_plan_info(int op, int dtype, int vec, int64_t T, int64_t C, int* protocol, int* tma,
                 int64_t* tile_rows, int64_t* n_chunks) {
    if (op < 0 || op >= (int)OP_COUNT || (dtype != LR_F32 && dtype != LR_BF16) || T < 1 || C < 1)
        return LR_ERR_INVALID_ARG;
    const bool v = vec != 0;
    // the same plan the entry points make (plan(), onepass_begin)
    const CarryPlan cp = carry_plan((Op)op, dtype, v, use_tma(dtype, v, T, C), T, C);
    if (protocol) *protocol = cp.mode;
    if (tma) *tma = cp.tma ? 1 : 0;
    if (tile_rows) *tile_rows = cp.ts.L;
    if (n_chunks) *n_chunks = cp.n_chunks;
    return LR_OK;
}

int lr_test_fail_after_enqueue(float* x, int64_t n, float value, uint64_t sleep_ns, void* stream) {
    if (n < 0 || (n > 0 && !x)) return LR_ERR_INVALID_ARG;
    GUARD;
    cudaStream_t s = (cudaStream_t)stream;
    DevWS* ws;
    TRY(get_ws(&ws));
    TRY(enter(*ws, s));
    Leave lv(*ws, s);
    k_test_sleep_fill<<<64, 256, 0, s>>>(x, n, value, sleep_ns);
    CK(cudaGetLastError());
    snprintf(g_cuda_msg, sizeof g_cuda_msg, "injected by lr_test_fail_after_enqueue");
    return LR_ERR_CUDA;  // as if a later launch of the call had failed
}

int lr_test_activations(const float* x, float* tanh_out, float* sigmoid_out, float* expm1_out,
                        int64_t n, void* stream) {
    GUARD;
    if (n < 0 || (n > 0 && (!x || !tanh_out || !sigmoid_out))) return LR_ERR_INVALID_ARG;
    if (n == 0) return LR_OK;
    const int64_t blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    k_test_act<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(x, tanh_out, sigmoid_out,
                                                                    expm1_out, n);
    CK(cudaGetLastError());
    return LR_OK;
}

int lr_test_lookback_timeout(uint32_t spin_limit, void* stream) {
    GUARD;
    cudaStream_t s = (cudaStream_t)stream;
    DevWS* ws;
    TRY(get_ws(&ws));
    // Chain protocol: both chain kernels (register and TMA-staged) on a problem
    // of two time chunks and one channel tile, each with one CTA that is handed
    // tile 1: it waits for the state after tile 0, which nobody publishes.
    // Look-back protocol: the same, tile 1 waits for tile 0's aggregate.
    // Cluster kernel: a two-chunk problem whose CTAs each expect one chunk
    // aggregate more than arrives.
    // Walker protocol: the register walker kernel (scalar path), the
    // warp-specialised one (vector path), the segmented walker kernel and its
    // consume-only form, on a long one-strip problem launched without walkers:
    // no entering state is ever published, so every consume's wait runs out.
    const int64_t C = tile_shape(OP_SCAN_FWD, LR_F32, true, CARRY_CHAIN).CW;
    const int64_t Tw = 8192;  // >= 128 chunks of both walker tile shapes
    if (!ws->test_buf) {
        CK(cudaMalloc(&ws->test_buf, (size_t)(3 * Tw * C) * sizeof(float)));
        CK(cudaMemset(ws->test_buf, 0, (size_t)(3 * Tw * C) * sizeof(float)));
        ws->bytes += 3 * Tw * C * (int64_t)sizeof(float);
    }
    char* buf = (char*)ws->test_buf;
    TRY(enter(*ws, s));
    Leave lv(*ws, s);
    for (int tma = 0; tma < 2; ++tma) {
        const int64_t T = 2 * tile_shape(OP_SCAN_FWD, LR_F32, true, tma ? TILE_TMA : CARRY_CHAIN).L;
        Geom g;
        Carry cr;
        TRY(plan(*ws, OP_SCAN_FWD, LR_F32, true, T, C, C, &g, &cr, s, tma, true));
        if (cr.mode != CARRY_CHAIN || cr.tma != tma) return LR_ERR_INVALID_ARG;
        g.max_grid = 1;
        g.ticket_base = 1;
        cr.spin_limit = spin_limit;
        const float* a = (const float*)buf;
        CK(launch_scan_fwd(LR_F32, true, a, a + Tw * C, nullptr, (float*)buf + 2 * Tw * C, g, cr,
                           s));
    }
    {  // look-back kernel
        const int64_t T = 2 * tile_shape(OP_SCAN_FWD, LR_F32, true, TILE_TMA).L;
        Geom g;
        Carry cr;
        TRY(plan(*ws, OP_SCAN_FWD, LR_F32, true, T, C, C, &g, &cr, s, 1, false, false));
        if (cr.mode != CARRY_LOOK) return LR_ERR_INVALID_ARG;
        g.max_grid = 1;
        g.ticket_base = 1;
        cr.spin_limit = spin_limit;
        const float* a = (const float*)buf;
        CK(launch_scan_fwd(LR_F32, true, a, a + Tw * C, nullptr, (float*)buf + 2 * Tw * C, g, cr,
                           s));
    }
    {  // cluster kernel: every CTA expects one chunk aggregate more than the CTAs before it send
        const int64_t T = 2 * tile_shape(OP_SCAN_FWD, LR_F32, true, TILE_CLUSTER).L;
        Geom g;
        Carry cr;
        TRY(plan(*ws, OP_SCAN_FWD, LR_F32, true, T, C, C, &g, &cr, s, 1));
        if (cr.mode != CARRY_CLUSTER) return LR_ERR_INVALID_ARG;
        g.ticket_base = 1;
        cr.spin_limit = spin_limit;
        const float* a = (const float*)buf;
        CK(launch_scan_fwd(LR_F32, true, a, a + Tw * C, nullptr, (float*)buf + 2 * Tw * C, g, cr, s));
    }
    for (int vec = 0; vec < 2; ++vec) {  // fp32 forward: register walker (scalar), warp-specialised (vector)
        Geom g;
        Carry cr;
        TRY(plan(*ws, OP_SCAN_FWD, LR_F32, vec == 1, Tw, C, C, &g, &cr, s, 0));
        if (cr.mode != CARRY_WALK || cr.tma) return LR_ERR_INVALID_ARG;
        cr.n_walk = 0;
        cr.spin_limit = spin_limit;
        CK(launch_scan_fwd(LR_F32, vec == 1, buf, buf + Tw * C * 4, nullptr, buf + 2 * Tw * C * 4, g,
                           cr, s));
    }
    {  // bf16 backward: the segmented walker
        Geom g;
        Carry cr;
        TRY(plan(*ws, OP_SCAN_BWD, LR_BF16, true, Tw, C, C, &g, &cr, s, 1));
        if (cr.mode != CARRY_WALK || !cr.tma) return LR_ERR_INVALID_ARG;
        cr.n_walk = 0;
        cr.spin_limit = spin_limit;
        const size_t n = (size_t)(Tw * C) * 2;  // bytes of one bf16 array
        CK(launch_scan_bwd(LR_BF16, true, buf, buf + n, nullptr, buf + 2 * n, buf + 3 * n, buf + 4 * n,
                           nullptr, g, cr, s));
    }
    {  // the consume-only segmented kernel: a DEER iteration whose aggregates
       // count as published, again without walker CTAs
        Geom g;
        Carry cr;
        TRY(plan(*ws, OP_DEER, LR_F32, true, Tw, C, C, &g, &cr, s, 1));
        if (cr.mode != CARRY_WALK || !cr.tma) return LR_ERR_INVALID_ARG;
        cr.n_walk = 0;
        cr.spin_limit = spin_limit;
        const float* z = (const float*)buf;  // zeros: w, u and the previous iterate
        const NextAgg nx{cr.agg, 0u, 1u, 0u};
        CK(launch_deer_iter(LR_F32, true, z, z, nullptr, z + Tw * C, (float*)buf + 2 * Tw * C,
                            ws->words + kWordSlots, nullptr, 0.f, nx, DeerSeq{nullptr, nullptr, nullptr}, g,
                            cr, s));
    }
    return lv.done();
}

}  // extern "C"
