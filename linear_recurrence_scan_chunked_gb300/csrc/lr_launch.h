// lr_launch.h -- host-side interface between the C ABI (lr_api.cu) and the
// kernel translation units.  Each operation exposes its tile shape (so the
// API can size the carry workspace) and a launcher that picks the
// template instance for the storage type and the vector / scalar path.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lr_common.cuh"

// Consume lag of the walker-protocol kernel, in rounds of tickets, and the
// L2 budget (MB) for the tiles parked between their two reads.
#ifndef LR_STREAM_LAG
#define LR_STREAM_LAG 2
#endif
#ifndef LR_STREAM_L2MB
#define LR_STREAM_L2MB 32
#endif
// The fp32 / bf16 forward scan's walker-protocol launches take the
// warp-specialised TMA kernel where it applies (0: the register kernel).
#ifndef LR_STREAM_WS
#define LR_STREAM_WS 1
#endif
// L2 budget (MB) of the segmented walker kernel: segments read twice.
#ifndef LR_SEG_L2MB
#define LR_SEG_L2MB 160
#endif
// The same sizing for the DEER iterations' segments (no second read).
#ifndef LR_SEG1_L2MB
#define LR_SEG1_L2MB 320
#endif

// The fused forward cells (SRU, LSTM) run the strip kernel with one barrier
// per tile (their backward kernels would not keep two CTAs per SM with the
// second buffer of warp aggregates).
// Warps per CTA of the DEER iterations' TMA-staged and walker kernels: four
// (16-row tiles, four CTAs per SM) keep the per-chunk barrier and the warps'
// prefix fold short; the iterations are bound by instruction issue, and
// 4-warp CTAs measured 2.5% faster than 8-warp ones.
#ifndef LR_DEER_NW
#define LR_DEER_NW 4
#endif
#ifndef LR_STRIP_ONEB
#define LR_STRIP_ONEB 1
#endif

// Register cap of the TMA-staged kernel: two CTAs of NW+1 = 9 warps per SM.
#ifndef LR_TMA_MAXNREG
#define LR_TMA_MAXNREG 112
#endif

namespace lrs {

struct TileShape {
    int L;    // time rows per tile
    int CW;   // channels per tile
    int threads;
};

enum Op {
    OP_SCAN_FWD = 0,
    OP_SCAN_BWD,
    OP_SRU_FWD,
    OP_SRU_BWD,
    OP_DEER,
    OP_DEER_BWD,
    OP_LSTM_FWD,
    OP_LSTM_BWD,
    OP_DEER_ODE,
    OP_COUNT
};

// Launch configuration of every kernel: NW warps per CTA, R rows per thread
// (tile = NW*R rows), VEC channels per lane (16-byte vectors on the vector
// path, one element on the scalar path), and for the TMA-staged chain kernel
// ST shared-memory stages.  The register chain kernel keeps two tiles in
// registers (the one being processed and the one being loaded), the walker
// kernel one; R is sized so that they fit in the registers of a thread at two
// CTAs per SM.  The TMA kernel keeps one tile in registers and ST in shared
// memory (about 96 KB of stages per CTA, two CTAs per SM).  One table, used
// both to instantiate the kernels and to size the workspace.
constexpr int TILE_TMA = 2;      // kcfg row of the TMA-staged chain kernel
constexpr int TILE_CLUSTER = 3;  // kcfg row of the cluster kernel
struct KCfg {
    int NW;
    int R;
    int ST;
};
constexpr KCfg kcfg(Op op, int dtype, int mode) {
    // bf16 holds two elements per register: twice the rows of fp32 (but the
    // DEER forms keep two fp32 values per element between their passes, J and
    // the right-hand side or the backward's two factors: the rows of fp32 for
    // both storage types).  The LSTM cell stages as many arrays per direction
    // as the SRU cell and takes its rows; DEER's ODE form takes the tanh
    // form's rows at eight warps per CTA (its heavier producer measured slower
    // with four).
    return mode == TILE_CLUSTER ? KCfg{8, 16, 0}  // 16 rows of 32 channels per warp, 128 per CTA
           : op == OP_DEER_ODE   ? KCfg{8, mode == CARRY_CHAIN ? 2 : 4, mode == TILE_TMA ? 3 : 0}
           : op == OP_DEER && dtype == 1 ? kcfg(OP_DEER, 0, mode)
           : op == OP_LSTM_FWD ? kcfg(OP_SRU_FWD, dtype, mode)
           : op == OP_LSTM_BWD ? kcfg(OP_SRU_BWD, dtype, mode)
           : op == OP_DEER_BWD ? KCfg{8, mode == CARRY_CHAIN ? 2 : 4, mode == TILE_TMA ? 3 : 0}
           : mode == CARRY_CHAIN
               ? (op == OP_SCAN_FWD ? KCfg{8, dtype == 1 ? 8 : 4, 0}
                  : op == OP_SCAN_BWD ? KCfg{8, dtype == 1 ? 4 : 2, 0}
                  : op == OP_SRU_FWD  ? KCfg{8, dtype == 1 ? 4 : 2, 0}
                  : op == OP_SRU_BWD  ? KCfg{8, dtype == 1 ? 2 : 1, 0}
                  :                     KCfg{8, dtype == 1 ? 4 : 2, 0})
           : mode == CARRY_WALK
               ? (op == OP_SCAN_FWD ? KCfg{8, 8, 0}
                  : op == OP_SCAN_BWD ? KCfg{8, dtype == 1 ? 8 : 4, 0}
                  : op == OP_SRU_FWD  ? KCfg{8, dtype == 1 ? 8 : 4, 0}
                  : op == OP_SRU_BWD  ? KCfg{8, dtype == 1 ? 4 : 2, 0}
                  : op == OP_DEER     ? KCfg{LR_DEER_NW, 4, 0}
                  :                     KCfg{8, dtype == 1 ? 8 : 4, 0})
               : (op == OP_SCAN_FWD ? KCfg{8, dtype == 1 ? 8 : 4, 3}
                  : op == OP_SCAN_BWD ? KCfg{8, dtype == 1 ? 8 : 4, 2}
                  : op == OP_SRU_FWD  ? KCfg{8, dtype == 1 ? 4 : 2, 3}
                  : op == OP_SRU_BWD  ? KCfg{8, dtype == 1 ? 4 : 2, 2}
                  : op == OP_DEER     ? KCfg{LR_DEER_NW, 4, 3}
                  :                     KCfg{8, dtype == 1 ? 8 : 4, 3});
}
// 4 channels per lane: 16-byte fp32 / 8-byte bf16 accesses, 128 channels per tile
constexpr int kvec(int dtype, bool vec) { return vec ? 4 : 1; }

// mode: CARRY_CHAIN, CARRY_WALK, TILE_TMA (chain protocol, TMA staging) or
// TILE_CLUSTER (tiles 32 channels wide on both paths: R rows of 32 channels
// per warp, held as VEC row groups)
inline TileShape tile_shape(Op op, int dtype, bool vec, int mode) {
    const KCfg k = kcfg(op, dtype, mode);
    return TileShape{k.NW * k.R, 32 * (mode == TILE_CLUSTER ? 1 : kvec(dtype, vec)), 32 * k.NW};
}

// The cluster kernel: at most this many time chunks (CTAs per cluster; above
// the portable 8, the launch opts in to Blackwell's 16), so problems of up to
// kClusterMax * 128 steps.  The scans have a cluster form; the cells and DEER
// keep their protocols.
constexpr int kClusterMax = 16;
constexpr int kClusterPortable = 8;
constexpr bool cluster_op(Op op) { return op == OP_SCAN_FWD || op == OP_SCAN_BWD; }

// The chain protocol stages its tiles with TMA when the vector path applies
// and the rows of the [T, C] sequence are 16-byte multiples (tensor-map
// strides) and at least one channel tile wide, with coordinates inside int32.  The tile height of the TMA kernel
// can differ from the register kernel's, so this choice, like the protocol,
// is fixed by the shape and the buffers' alignment of a call.
// The walker protocol runs the segmented TMA kernel when its tile is at least
// as tall as the register walker kernel's (per-chunk costs are paid twice
// there, once per pass); otherwise the register kernel with its taller tile.
constexpr bool seg_walk(Op op, int dtype) {
    return kcfg(op, dtype, TILE_TMA).NW * kcfg(op, dtype, TILE_TMA).R >=
           kcfg(op, dtype, CARRY_WALK).NW * kcfg(op, dtype, CARRY_WALK).R;
}

inline bool use_tma(int dtype, bool vec, int64_t T, int64_t C) {
    const int64_t es = dtype == 1 ? 2 : 4;
    return vec && (C * es) % 16 == 0 && C >= 128 && T < ((int64_t)1 << 30) &&
           C < ((int64_t)1 << 30);
}

// Which carry protocol a launch uses, its tile shape, and the packet storage
// it needs.  CLUSTER when every time chunk of a channel tile fits one
// thread-block cluster (the scans of up to kClusterMax * 128 steps: no packets
// at all).  WALK pays off once the chunk chain is long (a round trip per
// chunk level would dominate) and the channels are few enough for a handful
// of walker CTAs; LOOK when the problem is short enough for every tile to
// fold all the chunk aggregates before it (TMA path); otherwise CHAIN (the
// strip kernel for wide problems).  The choice depends on the shape only, so a
// given problem always gets the same association of its floating-point
// operations.
struct CarryPlan {
    int mode;          // CARRY_CHAIN / CARRY_WALK / CARRY_LOOK / CARRY_CLUSTER
    bool tma;          // CHAIN: a TMA-staged kernel runs it (strip / TMA chain)
    TileShape ts;      // tile shape of that protocol
    int64_t n_chunks;  // ceil(T / ts.L)
    uint32_t n_walk;   // walker CTAs
    int wv;            // channels per walker warp
    size_t inc_elems;  // state packets: n_chunks * C
    size_t agg_elems;  // aggregate packets (WALK, LOOK): 2 * n_chunks * C
};
constexpr int64_t kWalkMinChunks = 128;
// The look-back protocol reads, for a tile of chunk q, q aggregate packets
// per channel: about n_chunks^2 / 2 * 2 KB per channel tile in all.  It runs
// while n_chunks^2 * n_ct stays within this bound (~32 MB of L2 reads), i.e.
// where the chunk chain's one round trip per chunk level, not the bytes,
// would bound the launch.
constexpr int64_t kLookBudget = 32768;
// Channel strips from which the strip kernel runs a chain-protocol launch
// (one CTA per strip or more strips per CTA; fewer strips would leave SMs
// idle, and the chain kernel spreads the chunks of few strips over all SMs).
constexpr int64_t kStripMinStrips = 128;
constexpr int64_t kWalkMaxCtas = 32;

// The chain protocol's plan (TMA-staged or through registers).
inline CarryPlan chain_plan(Op op, int dtype, bool vec, bool tma, int64_t T, int64_t C) {
    CarryPlan p{};
    p.mode = CARRY_CHAIN;
    p.tma = tma && vec;
    p.ts = tile_shape(op, dtype, vec, p.tma ? TILE_TMA : CARRY_CHAIN);
    p.n_chunks = (T + p.ts.L - 1) / p.ts.L;
    p.n_walk = 0;
    p.wv = 0;
    p.inc_elems = (size_t)(p.n_chunks * C);
    p.agg_elems = 0;
    return p;
}

inline CarryPlan carry_plan(Op op, int dtype, bool vec, bool tma, int64_t T, int64_t C,
                            bool cluster = true) {
    CarryPlan p{};
    if (cluster && cluster_op(op)) {  // short problems: one cluster per channel tile
        const TileShape tk = tile_shape(op, dtype, vec, TILE_CLUSTER);
        const int64_t nk = (T + tk.L - 1) / tk.L;
        if (nk >= 1 && nk <= kClusterMax) {
            p.mode = CARRY_CLUSTER;
            p.tma = false;
            p.ts = tk;
            p.n_chunks = nk;
            p.n_walk = 0;
            p.wv = 0;
            p.inc_elems = 0;
            p.agg_elems = 0;
            return p;
        }
    }
    tma = tma && vec;
    // the TMA kernels (segmented walker, strip, TMA chain) use the TMA tile shape
    const int wmode = tma && seg_walk(op, dtype) ? TILE_TMA : CARRY_WALK;
    const TileShape tw = tile_shape(op, dtype, vec, wmode);
    const int64_t nw = (T + tw.L - 1) / tw.L;
    if (nw >= kWalkMinChunks) {
        const int wv = C <= 256 ? 1 : WALK_MAX_WV;  // spread the walkers' reads over more SMs
        const int64_t warps = (C + wv - 1) / wv;
        const int nwarp = kcfg(op, dtype, wmode).NW;
        const int64_t ctas = (warps + nwarp - 1) / nwarp;
        if (ctas * nwarp <= kWalkMaxCtas * 8) {  // at most 256 walker warps
            p.mode = CARRY_WALK;
            p.tma = wmode == TILE_TMA;  // segmented walker kernel, else the register one
            p.ts = tw;
            p.n_chunks = nw;
            p.n_walk = (uint32_t)ctas;
            p.wv = wv;
            p.inc_elems = (size_t)(nw * C);
            p.agg_elems = (size_t)(2 * nw * C);
            return p;
        }
    }
    if (tma) {
        const TileShape tt = tile_shape(op, dtype, vec, TILE_TMA);
        const int64_t nc = (T + tt.L - 1) / tt.L, nct = (C + tt.CW - 1) / tt.CW;
        if (nct < kStripMinStrips && nc <= 4096 && nc * nc * nct <= kLookBudget) {
            p.mode = CARRY_LOOK;
            p.tma = true;
            p.ts = tt;
            p.n_chunks = nc;
            p.n_walk = 0;
            p.wv = 0;
            p.inc_elems = 0;
            p.agg_elems = (size_t)(2 * nc * C);
            return p;
        }
    }
    return chain_plan(op, dtype, vec, tma, T, C);
}

// Grid of a persistent launch: every walker plus as many tile CTAs as can be
// resident at once (never more than there are tiles).
inline int sm_count() {
    static int sms[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& n_sm = sms[dev & 63];
    if (n_sm <= 0) {
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
        if (n_sm <= 0) n_sm = 1;
    }
    return n_sm;
}
inline uint32_t persist_grid(const Geom& g, const Carry& cr, int occ_per_sm) {
    const int n_sm = sm_count();
    const uint64_t want = (uint64_t)cr.n_walk + g.n_tiles;
    uint64_t cap = (uint64_t)occ_per_sm * (uint64_t)n_sm;
    if (cap < (uint64_t)cr.n_walk + 1) cap = (uint64_t)cr.n_walk + 1;
    uint64_t grid = want < cap ? want : cap;
    if (g.max_grid && grid > g.max_grid) grid = g.max_grid;
    return (uint32_t)grid;
}

cudaError_t launch_scan_fwd(int dtype, bool vec, const void* a, const void* b, const void* h0,
                            void* h, const Geom& g, const Carry& cr, cudaStream_t s);

cudaError_t launch_scan_bwd(int dtype, bool vec, const void* a, const void* h, const void* h0,
                            const void* dh, void* da, void* db, void* dh0, const Geom& g,
                            const Carry& cr, cudaStream_t s);

cudaError_t launch_sru_fwd(int dtype, bool vec, const void* xt, const void* uf, const void* ur,
                           const void* x, const float* bf, const float* br, const void* c0,
                           void* h, void* c, const Geom& g, const Carry& cr, cudaStream_t s);

// partials: [2][n_chunks][C] (forget, reset) fp32 scratch, followed by 2*C
// floats that launch_bias_reduce uses for its per-channel sums
cudaError_t launch_sru_bwd(int dtype, bool vec, const void* xt, const void* uf, const void* ur,
                           const void* x, const float* bf, const float* br, const void* c0,
                           const void* c, const void* dh, void* dxt, void* duf, void* dur,
                           void* dx, void* dc0, float* partials, const Geom& g,
                           const Carry& cr, cudaStream_t s);

// Per-feature sums of the per-tile partials [n_arr][n_chunks][C] (n_arr <= 4)
// into out[k] ([D] each), in a fixed order; the partials buffer must hold
// n_arr * C more floats after them for the per-channel sums.
struct BiasOut {
    float* o[4];
};
cudaError_t launch_bias_reduce(const float* partials, int64_t n_chunks, int n_arr, int64_t B,
                               int64_t D, BiasOut out, cudaStream_t s);

// DEER per-sequence stopping state (all nullptr: one test for the batch).
struct DeerSeq {
    uint32_t* resid;           // [B] this iteration's residual bits per sequence, zeroed
    const uint32_t* done;      // [B] nonzero: stopped
    const uint32_t* all_done;  // nonzero: every sequence stopped
};
// resid: one fp32 slot (as bits), zeroed before the launch, receives max|ynew-yold|.
// nx: the next iteration's segment aggregates (segmented walker kernel only;
// nx.agg == nullptr otherwise), and whether this launch's were published by
// the previous one (then cr.agg must point at them).
cudaError_t launch_deer_iter(int dtype, bool vec, const float* w, const void* u, const void* h0,
                             const void* yold, void* ynew, uint32_t* resid,
                             const uint32_t* prev_resid, float eps, const NextAgg& nx,
                             const DeerSeq& sq, const Geom& g, const Carry& cr, cudaStream_t s);
// After iteration k of a per-sequence solve: stop the sequences whose residual
// fell below eps (or is not finite), record K = k for them, set all_done when
// none runs.
cudaError_t launch_deer_seq_update(const uint32_t* resid, uint32_t* done, int32_t* iters,
                                   uint32_t* all_done, int64_t B, float eps, int k,
                                   cudaStream_t s);
// At the end of a per-sequence solve: copy into y the sequences whose last
// iterate is in ybuf (even K; `launched` for those that never stopped).
cudaError_t launch_deer_seq_gather(const void* ybuf, void* y, const int32_t* iters, int launched,
                                   int64_t T, int64_t C, int64_t D, int dtype, cudaStream_t s);

// LSTM cell: the four gate pre-activations (or their gradients), [T, C]
// each, and the four per-feature biases, [D] each.
struct LstmGates {
    const void* f;
    const void* i;
    const void* c;
    const void* o;
};
struct LstmBias {
    const float* f;
    const float* i;
    const float* c;
    const float* o;
};
cudaError_t launch_lstm_fwd(int dtype, bool vec, const LstmGates& z, const LstmBias& b,
                            const void* c0, void* h, void* c, const Geom& g, const Carry& cr,
                            cudaStream_t s);
// partials: [4][n_chunks][C] fp32 scratch (forget, input, candidate, output),
// followed by 4*C floats for launch_bias_reduce
cudaError_t launch_lstm_bwd(int dtype, bool vec, const LstmGates& z, const LstmBias& b,
                            const void* c0, const void* c, const void* dh, const LstmGates& dz,
                            void* dc0, float* partials, const Geom& g, const Carry& cr,
                            cudaStream_t s);

// DEER, ODE form: one iteration (dt: [T] step lengths; clamps: the
// iteration's clamp counter, zeroed before the launch).
cudaError_t launch_deer_ode_iter(int dtype, bool vec, const float* w, const void* u,
                                 const float* dt, const void* h0, const void* yold, void* ynew,
                                 uint32_t* resid, const uint32_t* prev_resid, float eps,
                                 unsigned long long* clamps, const NextAgg& nx, const Geom& g,
                                 const Carry& cr, cudaStream_t s);

// DEER backward: partials is [n_chunks][C] fp32 scratch (dw per tile),
// followed by C floats that launch_bias_reduce uses for its per-channel sums
cudaError_t launch_deer_bwd(int dtype, bool vec, const float* w, const void* y, const void* h0,
                            const void* dy, void* du, void* dh0, float* partials, const Geom& g,
                            const Carry& cr, cudaStream_t s);

}  // namespace lrs
