// lr_persist.cuh -- the persistent kernels shared by every operation:
//   k_strip  (wide problems: channel strips walked through time, TMA-staged;
//             a one-barrier-per-tile variant for operations that opt in),
//   k_seg    (long, narrow problems: walker protocol over segments, TMA-staged),
//   k_seg1   (k_seg's consume pass alone, for launches whose segment
//             aggregates the previous launch published: DEER iterations),
//   k_look   (short problems: every tile publishes its aggregate at once and
//             folds those of the chunks before it -- one round trip, not one
//             per chunk level; TMA-staged),
//   k_tchain (chain protocol, TMA-staged, for what is none of these),
//   k_wstream (walker protocol, warp-specialised: TMA-staged reduce and
//             consume rings, the forward scan's long, narrow problems),
//   k_stream (walker protocol through registers),
//   k_chain  (chain protocol through registers: scalar / unaligned paths),
// and launch_persist, which picks one for a call.
//
// An operation is a policy struct `Op` providing:
//   S, VEC, NW, R, REV, MINB      storage type, channels per lane, warps, rows
//                                 per thread, reverse time (backward scans),
//                                 resident CTAs per SM to compile for
//   IN_ARRAYS                     input arrays read per element
//   Params, Regs, Work, Smem, Acc kernel arguments, one tile's loaded data per
//                                 thread, values passed from aggregate() to
//                                 finish(), extra shared memory, per-thread
//                                 accumulators kept across tiles
//   init_ptr(p)                   state before the scan (nullable)
//   skip(p)                       the whole launch has nothing to do (checked
//                                 first by every CTA)
//   load(src, p, g, tc, regs)     the loads of one tile, from global memory or
//                                 from a TMA-staged tile (GlobalSrc / SmemSrc)
//   TMA_N, tma_shift, tma_extra, tma_arrays   the arrays staged by TMA
//                                 (lr_tma.cuh)
//   aggregate(p, g, tc, regs, w, A, B, side)  this thread's (A, B) over its R
//                                 rows in scan order; with side = true it also
//                                 writes the outputs that need no carry
//   finish(p, g, tc, regs, w, s, sm, acc)  output pass from the entering state s
//                                 (tc.acc_run / acc_flush: per-channel sums may
//                                 run in acc across a run of tiles, see TileCoord)
//   at_exit(p, sm, acc)           once per tile CTA after its last tile
// and optionally NEXT_AGG / next_agg(p) (lr_common.cuh: the next launch's
// aggregates, folded in finish) and STRIP_ONE_BARRIER.
#pragma once

#include <string.h>

#include <algorithm>

#include <type_traits>

#include "lr_launch.h"
#include "lr_tma.cuh"

namespace lrs {

// Order generic-proxy shared-memory accesses before later async-proxy (TMA)
// accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct TileCoord {
    int64_t q;       // chunk index in scan order
    int64_t tchunk;  // chunk index in time
    int64_t c;       // first channel of this lane
    int64_t cd;      // its feature index, c mod D (VEC divides D on the vector path)
    bool cok;        // the lane's channels are inside the problem
    int64_t t0;      // time of this thread's first row (scan order)
    // A run of tiles of the same channels in scan order goes through this CTA
    // (strip kernel with one strip per CTA: the whole strip; segmented walker
    // kernel: a segment's consume pass): per-channel sums may run in registers
    // across the run (Acc, acc_run) and be reduced once, on its last tile
    // (acc_flush).
    bool acc_run;
    bool acc_flush;
};

// Coordinates of the tile of chunk q (scan order) and channel tile j, for the
// rows of warp `warp` of the tile (by default the calling warp).
template <class Op>
__device__ __forceinline__ TileCoord tile_coord_qj(const Geom& g, uint32_t q, uint32_t j,
                                                   int warp = -1) {
    constexpr int L = Op::NW * Op::R, CW = 32 * Op::VEC;
    const int lane = threadIdx.x & 31;
    if (warp < 0) warp = threadIdx.x >> 5;
    TileCoord tc;
    tc.q = q;
    tc.c = (int64_t)j * CW + lane * Op::VEC;
    tc.cd = chan_feat(g, tc.c);
    tc.cok = tc.c < g.C;
    tc.tchunk = Op::REV ? g.n_chunks - 1 - tc.q : tc.q;
    tc.t0 = Op::REV ? tc.tchunk * L + (L - 1) - warp * Op::R : tc.tchunk * L + warp * Op::R;
    tc.acc_run = false;
    tc.acc_flush = false;
    return tc;
}

template <class Op>
__device__ __forceinline__ TileCoord tile_coord(const Geom& g, uint32_t tile) {
    return tile_coord_qj<Op>(g, tile / (uint32_t)g.n_ct, tile % (uint32_t)g.n_ct);
}

// Issue the global loads of one tile (register kernels).
template <class Op>
__device__ __forceinline__ void gload(const typename Op::Params& p, const Geom& g, uint32_t tile,
                                      typename Op::Regs& rg) {
    const TileCoord tc = tile_coord<Op>(g, tile);
    Op::load(GlobalSrc{g.C, tc.c}, p, g, tc, rg);
}

// The streaming kernel of the walker protocol.  Every CTA draws tickets; the
// first cr.n_walk tickets make walker CTAs.  Ticket X then
//   1. reduces tile X -- loads it, publishes its aggregate for the walkers and
//      keeps nothing,
//   2. consumes tile X - d_con: loads it again (now from L2, the reduce stage
//      brought it in d_con tickets earlier), combines the warp aggregates,
//      takes the state entering the tile from the walkers and writes the
//      outputs.
// A consume only waits for work of smaller tickets, and a reduce never waits,
// so every wait ends.  The walkers see each aggregate d_con tickets before any
// consumer needs the state it leads to, and HBM traffic stays one read of the
// inputs and one write of the outputs as long as the d_con tiles in flight fit
// in L2.
template <class Op>
__global__ void __launch_bounds__(Op::NW * 32, Op::MINB * 8 / Op::NW)
    k_stream(typename Op::Params p, Geom g, const Carry cr0, uint32_t d_con) {
    if (Op::skip(p)) {  // whole launch: before any ticket or barrier
        if (blockIdx.x == 0 && threadIdx.x == 0) retire_epoch(cr0);
        return;
    }
    constexpr int VEC = Op::VEC;
    __shared__ CarrySmem<VEC, Op::NW> sm;
    __shared__ typename Op::Smem xs;
    __shared__ uint32_t s_ticket, s_epoch;
    Carry cr = cr0;
    typename Op::Acc acc;
    Op::acc_init(acc);
    const uint32_t limit = cr.n_walk + g.n_tiles + d_con;
    bool tile_role = false;
    if (threadIdx.x == 0) {
        const uint32_t t = draw_ticket(cr);
        ticket_drawn(cr, g, t);
        s_ticket = t + g.ticket_base;
        s_epoch = cr.epoch;
    }
    __syncthreads();
    cr.epoch = s_epoch;
    uint32_t tk = s_ticket;
    while (true) {
        // the next ticket is drawn now and read after this one's work (a tile
        // CTA; a walker returns before it draws again)
        uint32_t next = 0;
        const bool draw = tk >= cr.n_walk && tk < limit;
        if (draw && threadIdx.x == 0) next = draw_ticket(cr);
        if (tk < cr.n_walk) {  // walker role
            walker<typename Op::S, Op::NW>(cr, g, tk, Op::init_ptr(p));
            return;
        }
        if (tk >= limit) break;
        tile_role = true;
        const uint32_t x = tk - cr.n_walk;
        const bool consume = x >= d_con && x - d_con < g.n_tiles;
        // the states entering the consumed tile, loaded now: usually they are
        // published long before the consume needs them, and then the carry
        // costs no round trip of its own
        u64 pre[VEC];
        if (consume && (threadIdx.x >> 5) == 0) {
            const TileCoord tc = tile_coord<Op>(g, x - d_con);
#pragma unroll
            for (int v = 0; v < VEC; ++v)
                pre[v] = (tc.q > 0 && tc.cok) ? ld_pkt(cr.inc + (tc.c + v) * g.n_chunks + tc.q - 1)
                                              : 0ull;
        }
        typename Op::Regs regs;
        typename Op::Work w;
        if (x < g.n_tiles) {  // reduce: publish the aggregate
            const TileCoord tc = tile_coord<Op>(g, x);
            Op::load(GlobalSrcHint{g.C, tc.c, l2_evict_last()}, p, g, tc, regs);
            float A[VEC], B[VEC];
            Op::aggregate(p, g, tc, regs, w, A, B, false);
            tile_publish_agg<VEC, Op::NW>(sm, A, B, cr, g, tc.q, tc.c, tc.cok);
        }
        if (consume) {  // the tile's last read
            const TileCoord tc = tile_coord<Op>(g, x - d_con);
            Op::load(GlobalSrcHint{g.C, tc.c, l2_evict_first()}, p, g, tc, regs);
            float A[VEC], B[VEC];
            Op::aggregate(p, g, tc, regs, w, A, B, true);
            float init[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) init[v] = 0.f;
            const typename Op::S* ip = Op::init_ptr(p);
            if (tc.q == 0 && (threadIdx.x >> 5) == 0 && ip != nullptr && tc.cok)
                load_vec<typename Op::S, VEC>(ip + tc.c, init);
            float s[VEC];
            tile_carry<VEC, Op::NW>(sm, A, B, init, s, cr, g, tc.q, tc.c, tc.cok, pre);
            Op::finish(p, g, tc, regs, w, s, xs, acc);
        }
        if (draw && threadIdx.x == 0) {
            ticket_drawn(cr, g, next);
            s_ticket = next + g.ticket_base;
        }
        __syncthreads();
        tk = s_ticket;
    }
    if (tile_role) Op::at_exit(p, xs, acc);
}

// Warp-specialised streaming kernel of the walker protocol (TMA staging).
// One CTA per SM; its warps take fixed roles and never wait for each other
// except through the rings between them:
//   * the reduce producer (one thread) draws the tickets.  Ticket X >= n_walk
//     stages tile X - n_walk into the reduce ring and queues tile
//     X - n_walk - d_con for consumption;
//   * NRW reducer warps fold a staged tile into its aggregate and publish it
//     for the walkers -- they wait for nothing but their data, so a tile's
//     aggregate follows its ticket by one HBM round trip, whatever the
//     consumers are waiting for;
//   * the consume producer (one thread) stages the queued tiles into the
//     consume ring (a re-read, normally from L2);
//   * NW consumer warps copy a staged tile into registers, hand the stage
//     back, take the state entering the tile from the walkers and write the
//     outputs;
//   * the walker warp is one of the protocol's walkers when the CTA's first
//     ticket is below n_walk (walker warp number = that ticket).
// A tile is staged as HS stages of L/HS rows (one box per array each), so
// that both rings hold several stages in the shared memory of one SM: STR
// reduce stages (the HBM reads in flight) and STC consume stages (the L2
// re-reads in flight; the consumers' side bounds the kernel, so it gets the
// larger share).  Warp 0 of the consumers loads the walkers' state packets
// of the next tile as soon as the consume producer has named it, a tile
// ahead of their use.
// Tickets below n_walk are only ever a CTA's first draw: a producer that
// started as a walker's CTA draws again only once n_walk tickets are out, so
// every walker is running before any tile is handed out, as in k_stream.  No
// wait is circular: reducers wait for data only, a consume waits for the
// aggregates of smaller tickets, and a producer blocked on a full queue holds
// no ticket whose tile it has not staged.  Every wait is bounded; a group
// that gives up decides to stop together, after its barrier.
#ifndef LR_WS_HS
#define LR_WS_HS 2
#endif
#ifndef LR_SEGRED
#define LR_SEGRED 1
#endif
#ifndef LR_WS_STR
#define LR_WS_STR 2
#endif
#ifndef LR_WS_STC
#define LR_WS_STC 4
#endif
#ifndef LR_WS_QD
#define LR_WS_QD 4
#endif
// Consume lag, in quarter rounds of the grid's tickets.  The second read of a
// tile hits L2 more often the sooner it follows the first (at full size DRAM
// reads were 1.31x the inputs at two rounds, 1.15x at half a round); the
// walkers keep up at half a round.
#ifndef LR_WS_LAG4
#define LR_WS_LAG4 2
#endif
constexpr uint32_t kWsNone = 0xffffffffu;  // end of a ring or queue

template <class Op>
struct WsLayout {
    static constexpr int NW = Op::NW, HS = LR_WS_HS, NRW = NW / HS;
    static constexpr int W_PR = NW + NRW, W_PC = W_PR + 1, W_WALK = W_PC + 1, NWARPS = W_WALK + 1;
    static constexpr int STR = LR_WS_STR, STC = LR_WS_STC, QD = LR_WS_QD;  // stages, queue slots
    static constexpr int SR = NW * Op::R / HS;  // rows per stage
    static_assert(NW % HS == 0, "a stage holds whole warps' rows");
    // bytes of array k in a stage, its offset, and the stage size
    __host__ __device__ static constexpr uint32_t arr_bytes(int k) {
        return (uint32_t)(SR + Op::tma_extra(k)) * 32u * Op::VEC * (uint32_t)sizeof(typename Op::S);
    }
    __host__ __device__ static constexpr uint32_t off(int k) {
        uint32_t o = 0;
        for (int j = 0; j < k; ++j) o += (arr_bytes(j) + 127u) & ~127u;
        return o;
    }
    static constexpr uint32_t SB = off(Op::TMA_N);
};

// Rows of a stage of k_wstream (row0: time of its first row).
template <class Op>
struct WsSrc {
    const unsigned char* stage;
    int64_t row0;
    int lane_e;
    template <class P, typename S>
    __device__ __forceinline__ void ld(P& pk, int k, const S*, int64_t t) const {
        constexpr int CW = 32 * Op::VEC;
        const int row = (int)(t - row0) - Op::tma_shift(k);
        pk.load_shared(reinterpret_cast<const S*>(stage + WsLayout<Op>::off(k)) + row * CW + lane_e);
    }
};

// One thread: issue the boxes of stage h of `tile` (one per array).
template <class Op>
__device__ __forceinline__ void ws_stage(const Geom& g, const TmaDesc& td, unsigned char* dst,
                                         uint64_t* full, uint32_t tile, int h, uint64_t pol) {
    using Ly = WsLayout<Op>;
    constexpr int L = Op::NW * Op::R, CW = 32 * Op::VEC;
    const int64_t q = tile / g.n_ct, j = tile % g.n_ct;
    const int64_t tchunk = Op::REV ? g.n_chunks - 1 - q : q;
    const int32_t x = (int32_t)(j * CW), y0 = (int32_t)(tchunk * L + h * Ly::SR);
    mbar_arrive_tx(full, td.tx_bytes);
#pragma unroll
    for (int a = 0; a < Op::TMA_N; ++a)
        if (td.present & (1u << a))
            tma_load_2d_hint(dst + Ly::off(a), &td.map[a], x, y0 + Op::tma_shift(a), full, pol);
}

// Ring bookkeeping of one producer thread: a stage whose last arming issued
// copies that nobody is known to have waited for keeps that use's parity
// (+1); before the thread exits it waits for those copies.
template <int ST>
struct WsRing {
    uint32_t k = 0;         // uses taken so far
    uint8_t pend[ST] = {};  // 0, or 1 + parity of the stage's last copy use
    // take the next use: its stage, once free (false: the wait ran out and
    // nothing was taken)
    __device__ __forceinline__ bool take(uint64_t* empty, const uint32_t* err, uint32_t& st,
                                         uint32_t& use) {
        st = k % ST;
        if (k >= ST && !mbar_wait(&empty[st], ((k / ST) - 1u) & 1u, err)) return false;
        pend[st] = 0;  // its previous copies were consumed
        use = k++;
        return true;
    }
    // a taken use was armed, with copies or without (an end marker)
    __device__ __forceinline__ void armed(uint32_t use, bool copies) {
        pend[use % ST] = copies ? (uint8_t)(1u + ((use / ST) & 1u)) : 0;
    }
    __device__ __forceinline__ void drain(uint64_t* full, const uint32_t* err) const {
        for (int i = 0; i < ST; ++i)
            if (pend[i]) mbar_wait(&full[i], pend[i] - 1u, err);
    }
};

template <class Op>
__global__ void __launch_bounds__(WsLayout<Op>::NWARPS * 32, 1)
    k_wstream(typename Op::Params p, Geom g, const Carry cr0, uint32_t d_con,
              const __grid_constant__ TmaDesc td) {
    if (Op::skip(p)) {  // whole launch: before any ticket or barrier
        if (blockIdx.x == 0 && threadIdx.x == 0) retire_epoch(cr0);
        return;
    }
    using Ly = WsLayout<Op>;
    constexpr int NW = Op::NW, VEC = Op::VEC, NRW = Ly::NRW, HS = Ly::HS, STR = Ly::STR,
                  STC = Ly::STC, QD = Ly::QD, SR = Ly::SR, L = Op::NW * Op::R, WPS = NW / HS;
    constexpr uint32_t SB = Ly::SB;
    extern __shared__ unsigned char dyn_smem[];
    unsigned char* ring_r = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + 127) & ~(uintptr_t)127);
    unsigned char* ring_c = ring_r + STR * SB;
    __shared__ float s_ra[2][NW][32][VEC], s_rb[2][NW][32][VEC];  // reduce: per-warp aggregates
    __shared__ float s_ca[2][NW][32][VEC], s_cb[2][NW][32][VEC];  // consume: per-warp aggregates
    __shared__ float s_cin[2][32][VEC];                           // state entering the consumed tile
    __shared__ typename Op::Smem xs;
    __shared__ __align__(8) uint64_t full_r[STR], empty_r[STR], full_c[STC], empty_c[STC];
    __shared__ __align__(8) uint64_t named_c[STC];  // s_ctile of the stage is written
    __shared__ __align__(8) uint64_t q_full[QD], q_empty[QD];
    __shared__ uint32_t s_rtile[STR], s_ctile[STC], s_q[QD];
    __shared__ uint32_t s_first, s_epoch, s_rabort, s_cabort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Carry cr = cr0;
    const uint32_t limit = cr.n_walk + g.n_tiles + d_con;
    if (threadIdx.x == 0) {
        for (int i = 0; i < STR; ++i) {
            mbar_init(&full_r[i], 1);
            mbar_init(&empty_r[i], NRW);  // every reducer warp reads every stage
        }
        for (int i = 0; i < STC; ++i) {
            mbar_init(&full_c[i], 1);
            mbar_init(&empty_c[i], WPS);  // the consumer warps whose rows it holds
            mbar_init(&named_c[i], 1);
        }
        for (int i = 0; i < QD; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
        }
        s_rabort = 0;
        s_cabort = 0;
        mbar_init_fence();
        const uint32_t t = draw_ticket(cr);
        ticket_drawn(cr, g, t);
        s_first = t + g.ticket_base;
        s_epoch = cr.epoch;
    }
    __syncthreads();
    cr.epoch = s_epoch;
    const uint32_t first = s_first;

    if (warp == Ly::W_WALK) {
        if (first < cr.n_walk) walker_warp<typename Op::S>(cr, g, first, Op::init_ptr(p));
        return;
    }

    if (warp == Ly::W_PR) {  // reduce producer
        if (lane != 0) return;
        const uint64_t pol = l2_evict_last();
        uint32_t t = first;
        bool ok = true;
        if (t < cr.n_walk) {
            // every walker role is taken before this CTA draws a tile ticket
            uint32_t spins = 0, sleep_ns = 0;
            while (true) {
                const uint32_t drawn = (uint32_t)ld_pkt(cr.tk) + g.ticket_base;
                if (drawn >= cr.n_walk) break;
                if (wait_step(cr, spins, sleep_ns, 256)) {
                    give_up(cr);
                    ok = false;
                    break;
                }
            }
            if (ok) {
                t = draw_ticket(cr);
                ticket_drawn(cr, g, t);
                t += g.ticket_base;
            }
        }
        WsRing<STR> rr;
        uint32_t kq = 0;
        while (ok && t < limit) {
            const uint32_t x = t - cr.n_walk;
            if (x < g.n_tiles) {
                for (int h = 0; h < HS && ok; ++h) {
                    uint32_t st, use;
                    if (!rr.take(empty_r, cr.err, st, use)) {
                        ok = false;
                        break;
                    }
                    s_rtile[st] = x;
                    ws_stage<Op>(g, td, ring_r + st * SB, &full_r[st], x, h, pol);
                    rr.armed(use, true);
                }
                if (!ok) {
                    give_up(cr);
                    break;
                }
            }
            if (x >= d_con && x - d_con < g.n_tiles) {
                const uint32_t sq = kq % QD;
                if (kq >= QD && !mbar_wait(&q_empty[sq], ((kq / QD) - 1u) & 1u, cr.err)) {
                    give_up(cr);
                    ok = false;
                    break;
                }
                s_q[sq] = x - d_con;
                mbar_arrive(&q_full[sq]);
                ++kq;
            }
            t = draw_ticket(cr);
            ticket_drawn(cr, g, t);
            t += g.ticket_base;
        }
        // the ends of the reduce ring (first stage of a tile) and of the queue;
        // after a timeout the other groups stop on the error word
        if (ok) {
            uint32_t st, use;
            if (rr.take(empty_r, cr.err, st, use)) {
                s_rtile[st] = kWsNone;
                mbar_arrive(&full_r[st]);
                rr.armed(use, false);
            }
            const uint32_t sq = kq % QD;
            if (kq < QD || mbar_wait(&q_empty[sq], ((kq / QD) - 1u) & 1u, cr.err)) {
                s_q[sq] = kWsNone;
                mbar_arrive(&q_full[sq]);
            }
        }
        rr.drain(full_r, cr.err);
        return;
    }

    if (warp == Ly::W_PC) {  // consume producer
        if (lane != 0) return;
        const uint64_t pol = l2_evict_first();
        WsRing<STC> rc;
        uint32_t kq = 0;
        bool ok = true;
        while (ok) {
            const uint32_t sq = kq % QD;
            if (!mbar_wait(&q_full[sq], (kq / QD) & 1u, cr.err)) break;
            const uint32_t y = s_q[sq];
            mbar_arrive(&q_empty[sq]);
            ++kq;
            for (int h = 0; h < HS; ++h) {  // the end goes to every stage of a tile
                uint32_t st, use;
                if (!rc.take(empty_c, cr.err, st, use)) {
                    ok = false;
                    break;
                }
                s_ctile[st] = y;
                mbar_arrive(&named_c[st]);
                if (y == kWsNone) {
                    mbar_arrive(&full_c[st]);
                    rc.armed(use, false);
                } else {
                    ws_stage<Op>(g, td, ring_c + st * SB, &full_c[st], y, h, pol);
                    rc.armed(use, true);
                }
            }
            if (y == kWsNone) break;
        }
        rc.drain(full_c, cr.err);
        return;
    }

    if (warp >= NW) {  // reducer warps: reducer rw takes the rows of warp rw + h*NRW in stage h
        const int rw = warp - NW;
        uint32_t par = 0;
        for (uint32_t k = 0;; ++k) {
            uint32_t x = kWsNone;
            bool bad = false;
#pragma unroll
            for (int h = 0; h < HS; ++h) {
                const uint32_t u = k * HS + h, st = u % STR;
                const bool got = __all_sync(0xffffffffu, mbar_wait(&full_r[st], (u / STR) & 1u, cr.err));
                if (!got) {
                    bad = true;
                    break;
                }
                if (h == 0) x = s_rtile[st];
                if (x == kWsNone) break;  // the end: a tile-less first stage
                const int vw = rw + h * NRW;
                const TileCoord tc = tile_coord_qj<Op>(g, x / (uint32_t)g.n_ct, x % (uint32_t)g.n_ct, vw);
                typename Op::Regs rg;
                Op::load(WsSrc<Op>{ring_r + st * SB, tc.tchunk * L + h * SR, lane * VEC}, p, g, tc, rg);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_r[st]);
                typename Op::Work w;
                float A[VEC], B[VEC];
                Op::aggregate(p, g, tc, rg, w, A, B, false);
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    s_ra[par][vw][lane][v] = A[v];
                    s_rb[par][vw][lane][v] = B[v];
                }
            }
            if (bad && lane == 0) {
                s_rabort = 1;
                atomicOr(cr.err, ERRBIT_TIMEOUT);
            }
            asm volatile("bar.sync 2, %0;" ::"r"(NRW * 32) : "memory");
            if (s_rabort != 0 || x == kWsNone) break;
            if (rw == 0) {
                const TileCoord tc = tile_coord_qj<Op>(g, x / (uint32_t)g.n_ct, x % (uint32_t)g.n_ct, 0);
                if (tc.cok && tc.q < g.n_chunks - 1) {
                    float TA[VEC], TB[VEC];
#pragma unroll
                    for (int v = 0; v < VEC; ++v) { TA[v] = 1.f; TB[v] = 0.f; }
#pragma unroll
                    for (int w = 0; w < NW; ++w)
#pragma unroll
                        for (int v = 0; v < VEC; ++v) {
                            const float a = s_ra[par][w][lane][v], b = s_rb[par][w][lane][v];
                            TB[v] = __fmaf_rn(a, TB[v], b);
                            TA[v] *= a;
                        }
#pragma unroll
                    for (int v = 0; v < VEC; ++v)
                        st_pkt2(cr.agg + 2 * ((tc.c + v) * g.n_chunks + tc.q), pkt(TA[v], cr.epoch),
                                pkt(TB[v], cr.epoch));
                }
            }
            par ^= 1u;
        }
        return;
    }

    // consumer warps: warp w's rows are in stage w / WPS of a tile
    typename Op::Acc acc;
    Op::acc_init(acc);
    const typename Op::S* ip = Op::init_ptr(p);
    const int h = warp / WPS;
    bool any = false;
    uint32_t par = 0;
    // Warp 0 loads the walkers' states for a tile one tile ahead: the tile's
    // number is in s_ctile as soon as the consume producer has named the
    // stage, long before its data lands, so the packets' round trip overlaps
    // the previous tile.
    u64 pre_next[VEC];
    auto peek = [&](uint32_t u) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) pre_next[v] = 0ull;
        const uint32_t st = u % STC;
        if (!mbar_wait(&named_c[st], (u / STC) & 1u, cr.err)) return;
        const uint32_t y = s_ctile[st];
        if (y == kWsNone) return;
        const TileCoord tn = tile_coord<Op>(g, y);
        if (tn.q > 0 && tn.cok) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) pre_next[v] = ld_pkt_cg(cr.inc + (tn.c + v) * g.n_chunks + tn.q - 1);
        }
    };
    if (warp == 0) peek(0);
    for (uint32_t k = 0;; ++k) {
        const uint32_t u = k * HS + h, st = u % STC;
        const bool got = __all_sync(0xffffffffu, mbar_wait(&full_c[st], (u / STC) & 1u, cr.err));
        const uint32_t y = got ? s_ctile[st] : kWsNone;
        if (!got && lane == 0) {
            s_cabort = 1;
            atomicOr(cr.err, ERRBIT_TIMEOUT);
        }
        TileCoord tc{};
        typename Op::Regs rg;
        if (y != kWsNone) {
            tc = tile_coord<Op>(g, y);
            Op::load(WsSrc<Op>{ring_c + st * SB, tc.tchunk * L + h * SR, lane * VEC}, p, g, tc, rg);
        }
        __syncwarp();
        if (lane == 0 && got) mbar_arrive(&empty_c[st]);  // copied into registers
        typename Op::Work w;
        if (y != kWsNone) {
            u64 pre[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) pre[v] = pre_next[v];
            if (warp == 0) peek((k + 1) * HS);
            float A[VEC], B[VEC];
            Op::aggregate(p, g, tc, rg, w, A, B, true);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                s_ca[par][warp][lane][v] = A[v];
                s_cb[par][warp][lane][v] = B[v];
            }
            if (warp == 0) {  // the walkers' state for this tile
                float cin[VEC];
#pragma unroll
                for (int v = 0; v < VEC; ++v) cin[v] = 0.f;
                if (tc.q == 0) {
                    if (ip != nullptr && tc.cok) load_vec<typename Op::S, VEC>(ip + tc.c, cin);
                } else {
                    bool ok = true;
#pragma unroll
                    for (int v = 0; v < VEC; ++v) {
                        ok = ok && (!tc.cok || pkt_ok(pre[v], cr.epoch));
                        cin[v] = pkt_val(pre[v]);
                    }
                    uint32_t spins = 0, sleep_ns = 0;
                    while (!__all_sync(0xffffffffu, ok)) {
                        if (__any_sync(0xffffffffu, wait_step(cr, spins, sleep_ns, kTileMaxSleepNs))) {
                            if (lane == 0) give_up(cr);
#pragma unroll
                            for (int v = 0; v < VEC; ++v) cin[v] = __int_as_float(0x7fc00000);
                            break;
                        }
                        ok = !tc.cok || get_states_strided<VEC>(cr.inc + tc.c * g.n_chunks + tc.q - 1,
                                                                g.n_chunks, cin, cr.epoch);
                    }
                }
#pragma unroll
                for (int v = 0; v < VEC; ++v) s_cin[par][lane][v] = cin[v];
            }
        }
        csync<NW>();
        if (s_cabort != 0 || y == kWsNone) break;
        any = true;
        float PA[VEC], PB[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { PA[v] = 1.f; PB[v] = 0.f; }
#pragma unroll
        for (int w2 = 0; w2 < NW - 1; ++w2) {
            if (w2 < warp) {
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    const float a = s_ca[par][w2][lane][v], b = s_cb[par][w2][lane][v];
                    PB[v] = __fmaf_rn(a, PB[v], b);
                    PA[v] *= a;
                }
            }
        }
        float s0[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) s0[v] = __fmaf_rn(PA[v], s_cin[par][lane][v], PB[v]);
        Op::finish(p, g, tc, rg, w, s0, xs, acc);
        par ^= 1u;
    }
    if (any) Op::at_exit(p, xs, acc);
}

// Whole consumer CTA: one tile whose data is in registers -- local scan,
// state entering the tile (chain protocol), output pass.
template <class Op>
__device__ __forceinline__ void tile_process(const typename Op::Params& p, const Geom& g,
                                             const Carry& cr, const TileCoord& tc,
                                             const typename Op::Regs& regs,
                                             CarrySmem<Op::VEC, Op::NW>& sm,
                                             typename Op::Smem& xs, typename Op::Acc& acc) {
    constexpr int VEC = Op::VEC;
    float A[VEC], B[VEC];
    typename Op::Work w;
    Op::aggregate(p, g, tc, regs, w, A, B, true);
    float init[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) init[v] = 0.f;
    const typename Op::S* ip = Op::init_ptr(p);
    if (tc.q == 0 && (threadIdx.x >> 5) == 0 && ip != nullptr && tc.cok)
        load_vec<typename Op::S, VEC>(ip + tc.c, init);
    float s[VEC];
    tile_carry<VEC, Op::NW>(sm, A, B, init, s, cr, g, tc.q, tc.c, tc.cok);
    Op::finish(p, g, tc, regs, w, s, xs, acc);
}

template <class Op>
__device__ __forceinline__ uint32_t chain_tile(const typename Op::Params& p, const Geom& g,
                                               const Carry& cr, uint32_t tile,
                                               const typename Op::Regs& regs,
                                               CarrySmem<Op::VEC, Op::NW>& sm,
                                               typename Op::Smem& xs, typename Op::Acc& acc,
                                               bool draw, uint32_t* s_ticket) {
    uint32_t next = 0;
    Carry c = cr;
    if (draw && threadIdx.x == 0) next = draw_ticket(c);  // latency hidden by the tile
    tile_process<Op>(p, g, cr, tile_coord<Op>(g, tile), regs, sm, xs, acc);
    if (draw && threadIdx.x == 0) {
        ticket_drawn(cr, g, next);
        *s_ticket = next + g.ticket_base;
    }
    __syncthreads();  // publishes the ticket; frees the carry smem for the next tile
    return draw ? *s_ticket : 0xffffffffu;
}

// Chain protocol through registers (scalar and unaligned paths): persistent
// CTAs walk their tiles in ticket order with two register sets.  While tile i
// is processed (local scan, wait for the state after the previous chunk,
// output pass) the loads of tile i+1 are in flight and the ticket of tile i+2
// is being drawn.  The chunk chain costs about one round trip per chunk level,
// hidden behind the tiles of the other channel tiles.
template <class Op>
__global__ void __launch_bounds__(Op::NW * 32, Op::MINB)
    k_chain(typename Op::Params p, Geom g, const Carry cr0) {
    if (Op::skip(p)) {  // whole launch: before any ticket or barrier
        if (blockIdx.x == 0 && threadIdx.x == 0) retire_epoch(cr0);
        return;
    }
    __shared__ CarrySmem<Op::VEC, Op::NW> sm;
    __shared__ typename Op::Smem xs;
    __shared__ uint32_t s_ticket, s_epoch;
    Carry cr = cr0;
    if (threadIdx.x == 0) {
        const uint32_t t = draw_ticket(cr);
        ticket_drawn(cr, g, t);
        s_ticket = t + g.ticket_base;
        s_epoch = cr.epoch;
    }
    __syncthreads();
    cr.epoch = s_epoch;
    uint32_t tk = s_ticket;
    const uint32_t limit = g.n_tiles;
    if (tk >= limit) return;
    typename Op::Acc acc;
    Op::acc_init(acc);
    typename Op::Regs r0, r1;
    uint32_t t0 = tk;
    gload<Op>(p, g, t0, r0);
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t t = draw_ticket(cr);
        ticket_drawn(cr, g, t);
        s_ticket = t + g.ticket_base;
    }
    __syncthreads();
    tk = s_ticket;
    while (true) {
        // tile t0 is loaded (r0); tk is the ticket of the next tile
        bool more = tk < limit;
        const uint32_t t1 = tk;
        if (more) gload<Op>(p, g, t1, r1);
        tk = chain_tile<Op>(p, g, cr, t0, r0, sm, xs, acc, more, &s_ticket);
        if (!more) break;
        more = tk < limit;
        t0 = tk;
        if (more) gload<Op>(p, g, t0, r0);
        tk = chain_tile<Op>(p, g, cr, t1, r1, sm, xs, acc, more, &s_ticket);
        if (!more) break;
    }
    Op::at_exit(p, xs, acc);
}

// Chain protocol with TMA staging.  Warp NW is the producer: its lane 0 draws
// the tickets (in order) and, for each tile, issues one box load per input
// array into the next free stage of a ring of ST stages.  Warps 0 .. NW-1
// consume the stages in the same order: copy the tile from shared memory into
// registers, hand the stage back, then scan it as the register kernel does.
// The consumers release a stage before they wait for the tile's carry, so up
// to ST tiles stream in while one waits.
//
// Every CTA consumes its tickets in ticket order and every drawn ticket
// belongs to a resident CTA, so the smallest unfinished tile can always
// finish: no wait is circular.  Every wait is bounded: a consumer that gives
// up on a stage sets the shared abort flag, and the consumers decide to stop
// together, after a barrier; the producer waits for its copies in flight
// before it exits.
// The producer also hands the consumers the launch's epoch (s_epoch, written
// before the first stage is armed: the consumers read it after their first
// completed wait).
template <class Op, int ST>
__device__ __forceinline__ void tma_produce(const Geom& g, Carry cr, const TmaDesc& td,
                                            unsigned char* ring, uint64_t* full, uint64_t* empty,
                                            uint32_t* s_tile, uint32_t* s_epoch) {
    constexpr int L = Op::NW * Op::R, CW = 32 * Op::VEC;
    constexpr uint32_t SB = tma_stage_bytes<Op>();
    uint32_t k = 0;          // stage uses so far
    bool last_plain = false; // use k was the final (tile-less) arrival
    for (;; ++k) {
        const uint32_t st = k % ST;
        const uint32_t t = draw_ticket(cr);  // latency overlaps the wait below
        ticket_drawn(cr, g, t);
        if (k == 0) *s_epoch = cr.epoch;
        if (k >= ST && !mbar_wait(&empty[st], ((k / ST) - 1u) & 1u, cr.err)) {
            give_up(cr);
            break;
        }
        const uint32_t tile = t + g.ticket_base;
        s_tile[st] = tile;
        if (tile >= g.n_tiles) {
            mbar_arrive(&full[st]);
            last_plain = true;
            break;
        }
        mbar_arrive_tx(&full[st], td.tx_bytes);
        const int64_t q = tile / g.n_ct, j = tile % g.n_ct;
        const int64_t tchunk = Op::REV ? g.n_chunks - 1 - q : q;
        const int32_t x = (int32_t)(j * CW), y0 = (int32_t)(tchunk * L);
        unsigned char* dst = ring + st * SB;
#pragma unroll
        for (int a = 0; a < Op::TMA_N; ++a)
            if (td.present & (1u << a))
                tma_load_2d(dst + tma_off<Op>(a), &td.map[a], x, y0 + Op::tma_shift(a), &full[st]);
    }
    // Uses [k - ST + last_plain, k) may still have copies in flight (the stage
    // of use k - ST was handed back before a final arrival on it).
    const uint32_t lo = k + (last_plain ? 1u : 0u) > ST ? k + (last_plain ? 1u : 0u) - ST : 0u;
    for (uint32_t i = lo; i < k; ++i) mbar_wait(&full[i % ST], (i / ST) & 1u, cr.err);
}

template <class Op, int ST>
__global__ void __maxnreg__(LR_TMA_MAXNREG)
    k_tchain(typename Op::Params p, Geom g, const Carry cr0, const __grid_constant__ TmaDesc td) {
    if (Op::skip(p)) {  // whole launch: before any ticket or barrier
        if (blockIdx.x == 0 && threadIdx.x == 0) retire_epoch(cr0);
        return;
    }
    constexpr int NW = Op::NW, VEC = Op::VEC, L = Op::NW * Op::R;
    constexpr uint32_t SB = tma_stage_bytes<Op>();
    extern __shared__ unsigned char dyn_smem[];
    // TMA destinations: 128-byte aligned (the launch adds 128 bytes of slack)
    unsigned char* ring = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + 127) & ~(uintptr_t)127);
    __shared__ CarrySmem<VEC, NW> sm;
    __shared__ typename Op::Smem xs;
    __shared__ __align__(8) uint64_t full[ST], empty[ST];
    __shared__ uint32_t s_tile[ST];
    __shared__ uint32_t s_abort, s_epoch;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Carry cr = cr0;
    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NW);
        }
        s_abort = 0;
        mbar_init_fence();
    }
    __syncthreads();
    if (warp == NW) {
        if (lane == 0) tma_produce<Op, ST>(g, cr, td, ring, full, empty, s_tile, &s_epoch);
        return;
    }
    typename Op::Acc acc;
    Op::acc_init(acc);
    for (uint32_t k = 0;; ++k) {
        const uint32_t st = k % ST;
        if (!mbar_wait(&full[st], (k / ST) & 1u, cr.err)) {
            s_abort = 1;
            atomicOr(cr.err, ERRBIT_TIMEOUT);
        }
        csync<NW>();  // the decision below is the same in every consumer
        cr.epoch = s_epoch;
        const uint32_t tile = s_tile[st];
        if (s_abort != 0 || tile >= g.n_tiles) break;
        const TileCoord tc = tile_coord<Op>(g, tile);
        typename Op::Regs regs;
        Op::load(SmemSrc<Op>{ring + st * SB, tc.tchunk * L, lane * VEC}, p, g, tc, regs);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        tile_process<Op>(p, g, cr, tc, regs, sm, xs, acc);
    }
    Op::at_exit(p, xs, acc);
}


// Look-back kernel (LOOK protocol; short problems whose chunk chain would
// cost one L2 round trip per chunk level).  The tiles are staged by TMA as in
// the TMA chain kernel (producer warp, tickets in scan order).  A tile
//   1. folds its rows into its aggregate and publishes it at once (before it
//      waits for anything): packets agg[q][c] = (A, B) of chunk q;
//   2. looks back over every chunk before it: warp w folds the aggregates of
//      its share [q*w/NW, q*(w+1)/NW) of chunks 0 .. q-1 (issued as one batch
//      of loads per LOOK_PB chunks, polled until they carry this launch's
//      epoch), and the state entering the tile is h0 carried through the NW
//      shares in order;
//   3. re-reads its rows from the stage and writes its outputs.
// Every chunk's aggregate is published before its tile waits, so once the
// tiles of a wave have reduced their rows, each wait costs one round trip to
// L2 instead of one per chunk level, and no chunk waits for another's state.
// The association of every operation is fixed by (q, NW): the result is
// bitwise reproducible.  The look-back reads q * 16 bytes per channel, which
// bounds the protocol to problems with few chunks (the launch plan).
#ifndef LR_LOOK_PB
#define LR_LOOK_PB 4
#endif
#ifndef LR_LOOK_PDL
#define LR_LOOK_PDL 1
#endif
constexpr int LOOK_PB = LR_LOOK_PB;  // preceding chunks per warp per batch of loads

// Warp-level: the fold of the aggregates of chunks [lo, hi) for this lane's
// channels, in chunk order.  Polls until every packet carries the launch's
// epoch; a wait that runs out gives NaN (and records the error).
template <int VEC>
__device__ __forceinline__ void look_fold(const Carry& cr, const Geom& g, uint32_t lo, uint32_t hi,
                                          int64_t c, bool cok, float (&RA)[VEC], float (&RB)[VEC]) {
    constexpr int PB = LOOK_PB;
#pragma unroll
    for (int v = 0; v < VEC; ++v) { RA[v] = 1.f; RB[v] = 0.f; }
    uint32_t spins = 0, sleep_ns = 0;
    bool dead = false;
    for (uint32_t p0 = lo; p0 < hi; p0 += PB) {
        const uint32_t n = hi - p0 < (uint32_t)PB ? hi - p0 : (uint32_t)PB;
        u64 pk[PB][VEC][2];
        bool okk[PB];
#pragma unroll
        for (int k = 0; k < PB; ++k) {
            okk[k] = !cok || (uint32_t)k >= n;
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                pk[k][v][0] = pk[k][v][1] = 0;
                if (!okk[k]) ld_pkt2(cr.agg + 2 * ((int64_t)(p0 + k) * g.C + c + v), pk[k][v][0], pk[k][v][1]);
            }
        }
        while (!dead) {
            bool all = true;
#pragma unroll
            for (int k = 0; k < PB; ++k) {
                if (!okk[k]) {
                    bool ok = true;
#pragma unroll
                    for (int v = 0; v < VEC; ++v)
                        ok = ok && pkt_ok(pk[k][v][0], cr.epoch) && pkt_ok(pk[k][v][1], cr.epoch);
                    okk[k] = ok;
                }
                all = all && okk[k];
            }
            if (__all_sync(0xffffffffu, all)) break;
            if (__any_sync(0xffffffffu, wait_step(cr, spins, sleep_ns, kTileMaxSleepNs))) {
                if ((threadIdx.x & 31) == 0) give_up(cr);
                dead = true;
                break;
            }
#pragma unroll
            for (int k = 0; k < PB; ++k)  // re-poll what was not visible
                if (!okk[k])
#pragma unroll
                    for (int v = 0; v < VEC; ++v)
                        ld_pkt2(cr.agg + 2 * ((int64_t)(p0 + k) * g.C + c + v), pk[k][v][0], pk[k][v][1]);
        }
        if (dead) break;
#pragma unroll
        for (int k = 0; k < PB; ++k)
            if ((uint32_t)k < n)
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    const float a = pkt_val(pk[k][v][0]);
                    RB[v] = __fmaf_rn(a, RB[v], pkt_val(pk[k][v][1]));
                    RA[v] *= a;
                }
    }
    if (dead) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) RA[v] = RB[v] = __int_as_float(0x7fc00000);
    }
}

// Thread 0 of a look-back CTA: issue the boxes of `tile` into stage st.
template <class Op>
__device__ __forceinline__ void look_load(const Geom& g, const TmaDesc& td, unsigned char* ring,
                                          uint64_t* full, uint32_t tile, uint32_t st) {
    constexpr int L = Op::NW * Op::R, CW = 32 * Op::VEC;
    const int64_t q = tile / g.n_ct, j = tile % g.n_ct;
    const int64_t tchunk = Op::REV ? g.n_chunks - 1 - q : q;
    const int32_t x = (int32_t)(j * CW), y0 = (int32_t)(tchunk * L);
    mbar_arrive_tx(&full[st], td.tx_bytes);
    unsigned char* dst = ring + st * tma_stage_bytes<Op>();
#pragma unroll
    for (int a = 0; a < Op::TMA_N; ++a)
        if (td.present & (1u << a))
            tma_load_2d(dst + tma_off<Op>(a), &td.map[a], x, y0 + Op::tma_shift(a), &full[st]);
}

// Thread 0 of a look-back CTA: draw the next ticket (tile, or past the end)
// into s_tile[st] and, for a tile, issue its boxes into stage st.
template <class Op>
__device__ __forceinline__ void look_issue(Carry& cr, const Geom& g, const TmaDesc& td,
                                           unsigned char* ring, uint64_t* full, uint32_t* s_tile,
                                           uint32_t st) {
    const uint32_t t = draw_ticket(cr);
    ticket_drawn(cr, g, t);
    const uint32_t tile = t + g.ticket_base;
    s_tile[st] = tile;
    if (tile < g.n_tiles) look_load<Op>(g, td, ring, full, tile, st);
}

// No producer warp: thread 0 draws the tickets (in order) and issues each
// tile's boxes, ST stages ahead, so that two CTAs of NW warps fit an SM and a
// problem of up to two tiles per SM runs in one wave.
//
// When the host sized the grid to one tile per CTA (g.n_draws == gridDim.x),
// the tile is the block index and its boxes are issued as soon as the kernel
// before has completed: no ticket stands between the dependency wait and the
// load, and the CTAs do not queue on one atomic before they start.  The epoch
// comes from a plain load of the ticket word, issued beside the boxes; each CTA
// draws one arrival ticket on the same word once it has published its
// aggregate (after that load, in the word's coherence order, and off the path
// of the other CTAs' epoch loads), and the last arrival retires the epoch when
// its CTA ends.  A tile waits only for tiles of smaller block index, which the
// hardware dispatches first; every one of them is resident in the same wave.
template <class Op, int ST>
__global__ void __launch_bounds__(Op::NW * 32, Op::MINB * 8 / Op::NW)
    k_look(typename Op::Params p, Geom g, const Carry cr0, const __grid_constant__ TmaDesc td) {
    constexpr int NW = Op::NW, VEC = Op::VEC, L = Op::NW * Op::R;
    constexpr uint32_t SB = tma_stage_bytes<Op>();
    extern __shared__ unsigned char dyn_smem[];
    unsigned char* ring = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + 127) & ~(uintptr_t)127);
    // warp aggregates of the tile, then (after a barrier) each warp's fold
    // of its share of the preceding chunks
    __shared__ StripSmem<VEC, NW> sm;
    __shared__ typename Op::Smem xs;
    __shared__ __align__(8) uint64_t full[ST];
    __shared__ uint32_t s_tile[ST];
    __shared__ uint32_t s_abort, s_epoch;
    // Before the dependency wait, only what the kernel before cannot have
    // written: the stage barriers and the tensor maps (kernel parameters).
    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) mbar_init(&full[i], 1);
        s_abort = 0;
        mbar_init_fence();
#pragma unroll
        for (int a = 0; a < Op::TMA_N; ++a)
            if (td.present & (1u << a)) tma_prefetch_desc(&td.map[a]);
    }
    // Launched as a programmatic dependent of the kernel before it: its CTAs
    // may be scheduled while that kernel still runs, and wait here until it
    // has completed and its writes are visible (a no-op without a
    // predecessor).  The next kernel may be scheduled as soon as this one runs.
    griddep_wait();
    griddep_launch_dependents();
    if (Op::skip(p)) {  // whole launch: before any ticket or barrier
        if (blockIdx.x == 0 && threadIdx.x == 0) retire_epoch(cr0);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool one = g.n_draws == gridDim.x;  // one tile per CTA, in block order
    Carry cr = cr0;
    bool drawing = true;     // thread 0: no ticket past the end drawn yet
    uint32_t issued = 0;     // thread 0: stage uses whose ticket was drawn
    unsigned long long arrival = 0;  // thread 0, one tile per CTA: the arrival draw
    bool arrived = false;
    if (threadIdx.x == 0) {
        if (one) {
            const uint32_t tile = blockIdx.x + g.ticket_base;
            s_tile[0] = tile;
            if (tile < g.n_tiles) look_load<Op>(g, td, ring, full, tile, 0);
            issued = 1;
            drawing = false;
            cr.epoch = epoch_after((uint32_t)(ld_pkt(cr.tk) >> 32));
        } else {
            for (; issued < (uint32_t)ST && drawing; ++issued) {
                look_issue<Op>(cr, g, td, ring, full, s_tile, issued);
                if (s_tile[issued] >= g.n_tiles) drawing = false;
            }
        }
        for (uint32_t i = issued; i < (uint32_t)ST; ++i) s_tile[i] = 0xffffffffu;
        s_epoch = cr.epoch;
    }
    __syncthreads();
    cr.epoch = s_epoch;
    typename Op::Acc acc;
    Op::acc_init(acc);
    uint32_t k = 0;
    for (;; ++k) {
        const uint32_t st = k % ST;
        const uint32_t tile = s_tile[st];
        if (tile >= g.n_tiles) break;  // uniform: s_tile is written before a barrier
        if (!mbar_wait(&full[st], (k / ST) & 1u, cr.err)) s_abort = 1;
        csync<NW>();  // uniform stop decision
        if (s_abort != 0) break;
        const TileCoord tc = tile_coord<Op>(g, tile);
        const SmemSrc<Op> src{ring + st * SB, tc.tchunk * L, lane * VEC};
        float A[VEC], B[VEC];
        {
            typename Op::Regs regs;
            typename Op::Work w;
            Op::load(src, p, g, tc, regs);
            Op::aggregate(p, g, tc, regs, w, A, B, false);
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            sm.a[warp][lane][v] = A[v];
            sm.b[warp][lane][v] = B[v];
        }
        csync<NW>();
        // 1. the tile's aggregate, published before any wait
        if (warp == 0 && tc.cok && tc.q < g.n_chunks - 1) {
            float TA[VEC], TB[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) { TA[v] = 1.f; TB[v] = 0.f; }
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2)
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    const float a = sm.a[w2][lane][v];
                    TB[v] = __fmaf_rn(a, TB[v], sm.b[w2][lane][v]);
                    TA[v] *= a;
                }
#pragma unroll
            for (int v = 0; v < VEC; ++v)
                st_pkt2(cr.agg + 2 * (tc.q * g.C + tc.c + v), pkt(TA[v], cr.epoch), pkt(TB[v], cr.epoch));
        }
        if (one && threadIdx.x == 0 && !arrived) {  // after the publish: off the loads' path
            arrival = atomicAdd(reinterpret_cast<unsigned long long*>(cr.tk), 1ull);
            arrived = true;
        }
        // the warps before this one within the tile, as one affine map
        float PA[VEC], PB[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { PA[v] = 1.f; PB[v] = 0.f; }
#pragma unroll
        for (int w2 = 0; w2 < NW - 1; ++w2)
            if (w2 < warp)
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    const float a = sm.a[w2][lane][v];
                    PB[v] = __fmaf_rn(a, PB[v], sm.b[w2][lane][v]);
                    PA[v] *= a;
                }
        // the state before the first chunk, loaded now so that its round trip
        // runs beside the look-back
        float s[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) s[v] = 0.f;
        const typename Op::S* ip = Op::init_ptr(p);
        if (ip != nullptr && tc.cok) load_vec<typename Op::S, VEC>(ip + tc.c, s);
        csync<NW>();  // sm is free for the look-back
        // 2. this warp's share of the preceding chunks
        const uint32_t q = (uint32_t)tc.q;
        const uint32_t lo = (uint32_t)(((uint64_t)q * warp) / NW);
        const uint32_t hi = (uint32_t)(((uint64_t)q * (warp + 1)) / NW);
        {
            float RA[VEC], RB[VEC];
            look_fold<VEC>(cr, g, lo, hi, tc.c, tc.cok, RA, RB);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                sm.a[warp][lane][v] = RA[v];
                sm.b[warp][lane][v] = RB[v];
            }
        }
        csync<NW>();
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2)
            if ((uint64_t)q * (w2 + 1) / NW > (uint64_t)q * w2 / NW)  // a non-empty share
#pragma unroll
                for (int v = 0; v < VEC; ++v) s[v] = __fmaf_rn(sm.a[w2][lane][v], s[v], sm.b[w2][lane][v]);
#pragma unroll
        for (int v = 0; v < VEC; ++v) s[v] = __fmaf_rn(PA[v], s[v], PB[v]);
        // 3. the outputs, from the rows still in the stage
        {
            typename Op::Regs regs;
            typename Op::Work w;
            float A2[VEC], B2[VEC];
            Op::load(src, p, g, tc, regs);
            Op::aggregate(p, g, tc, regs, w, A2, B2, true);
            Op::finish(p, g, tc, regs, w, s, xs, acc);
        }
        // every warp has read the stage and sm: thread 0 refills the stage
        // with the tile ST uses ahead (the next loop top reads s_tile after
        // this barrier)
        csync<NW>();
        if (threadIdx.x == 0) {
            if (drawing) {
                fence_proxy_async_smem();  // the generic reads of the stage before the async refill
                look_issue<Op>(cr, g, td, ring, full, s_tile, st);
                if (s_tile[st] >= g.n_tiles) drawing = false;
                ++issued;
            } else {
                s_tile[st] = 0xffffffffu;
            }
        }
        csync<NW>();
    }
    Op::at_exit(p, xs, acc);
    if (threadIdx.x == 0) {
        // after an early stop: copies still in flight land first
        for (uint32_t i = k; i < issued; ++i)
            if (s_tile[i % ST] < g.n_tiles) mbar_wait(&full[i % ST], (i / ST) & 1u, cr.err);
        if (one) {  // the last arrival retires the epoch
            if (!arrived) arrival = atomicAdd(reinterpret_cast<unsigned long long*>(cr.tk), 1ull);
            ticket_drawn(cr, g, (uint32_t)arrival);
        }
    }
}

// Cluster kernel (short problems): the CTAs of one thread-block cluster take
// the time chunks of one 32-channel tile, chunk q on the CTA of rank q.  Each
// CTA loads its rows into registers and forms its chunk's aggregate (the
// composition of the affine maps of its rows); its warps send it, with
// asynchronous stores, into the shared memory of every CTA after it in the
// cluster (one warp per receiver), where the stores count their bytes on that
// CTA's barrier.  A CTA of rank q waits until the q aggregates before its own
// have landed, folds them in chunk order into the state that enters its chunk,
// and writes its outputs.
// Nothing goes through global memory but the inputs and outputs: no packets,
// tickets or epochs, and no CTA waits for another cluster, so clusters may run
// in any order and any number of waves.
//
// Thread layout: a row of the tile is 32 channels, held by 32 / VEC lanes
// (VEC channels each), so a warp holds VEC row groups of R consecutive rows:
// lane l takes channels (l mod 32/VEC) * VEC and row group l / (32/VEC).  The
// groups of a warp are composed by a shuffle scan, the warps through shared
// memory.  The association of every operation is fixed by the chunk, warp and
// lane indices: the result is bitwise reproducible.
template <class Op, int CL>
__global__ void __launch_bounds__(Op::NW * 32, Op::MINB)
    k_cluster(typename Op::Params p, Geom g, const Carry cr) {
    constexpr int NW = Op::NW, VEC = Op::VEC, R = Op::R;
    constexpr int LPR = 32 / VEC;        // lanes per row
    constexpr int RG = VEC;              // row groups per warp
    constexpr int L = NW * RG * R;       // rows per CTA
    constexpr uint32_t kAggBytes = 32 * 8;  // one chunk's aggregate: (A, B) per channel
    static_assert(LPR * VEC == 32, "a row is 32 channels");
    static_assert(Op::RG == RG, "the op is instantiated for this kernel's row groups");
    // skip depends on the arguments only: the whole launch returns here,
    // before any barrier
    if (Op::skip(p)) return;
    __shared__ StripSmem<VEC, NW> sm;           // the warps' aggregates of this chunk
    __shared__ __align__(16) float2 cab[CL][32];  // (A, B) of the chunks before it
    __shared__ __align__(8) uint64_t cbar;      // counts their bytes
    __shared__ typename Op::Smem xs;
    if (threadIdx.x == 0) {
        mbar_init(&cbar, 1);
        mbar_init_fence();
    }
    // the first cluster barrier phase: no CTA stores into another before that
    // one runs and has initialised its barrier
    cluster_arrive_relaxed();
    // a programmatic dependent launch, as k_look
    griddep_wait();
    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cq = lane % LPR, rg = lane / LPR;
    const uint32_t q = cluster_rank(), n = cluster_ctas();
    // the bytes of the q chunk aggregates before this one (g.ticket_base adds
    // chunks that never come: the timeout test)
    if (threadIdx.x == 0) mbar_arrive_tx(&cbar, (q + g.ticket_base) * kAggBytes);
    TileCoord tc;
    tc.q = q;
    tc.tchunk = Op::REV ? g.n_chunks - 1 - (int64_t)q : (int64_t)q;
    {
        const int vb = warp * RG + rg;  // row block of R rows, in scan order
        tc.t0 = Op::REV ? tc.tchunk * L + (L - 1) - vb * R : tc.tchunk * L + vb * R;
    }
    tc.c = (int64_t)(blockIdx.x / n) * 32 + cq * VEC;
    tc.cd = chan_feat(g, tc.c);
    tc.cok = tc.c < g.C;
    tc.acc_run = false;
    tc.acc_flush = false;
    float s[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) s[v] = 0.f;
    const typename Op::S* ip = Op::init_ptr(p);
    if (ip != nullptr && tc.cok) load_vec<typename Op::S, VEC>(ip + tc.c, s);
    typename Op::Regs regs;
    typename Op::Work w;
    typename Op::Acc acc;
    Op::acc_init(acc);
    Op::load(GlobalSrc{g.C, tc.c}, p, g, tc, regs);
    // the row groups before this one within the warp (exclusive), and the
    // warp's aggregate (inclusive, on the last group)
    float EA[VEC], EB[VEC];
    {
        float IA[VEC], IB[VEC];
        Op::aggregate(p, g, tc, regs, w, IA, IB, false);
#pragma unroll
        for (int off = LPR; off < 32; off *= 2)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float ua = __shfl_up_sync(0xffffffffu, IA[v], off);
                const float ub = __shfl_up_sync(0xffffffffu, IB[v], off);
                if (lane >= off) {  // this group after the ones before it
                    IB[v] = __fmaf_rn(IA[v], ub, IB[v]);
                    IA[v] *= ua;
                }
            }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            EA[v] = RG > 1 ? __shfl_up_sync(0xffffffffu, IA[v], LPR) : 1.f;
            EB[v] = RG > 1 ? __shfl_up_sync(0xffffffffu, IB[v], LPR) : 0.f;
            if (rg == 0) { EA[v] = 1.f; EB[v] = 0.f; }
        }
        if (rg == RG - 1)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                sm.a[warp][cq][v] = IA[v];
                sm.b[warp][cq][v] = IB[v];
            }
    }
    csync<NW>();
    cluster_wait();  // the first phase
    // the chunk's aggregate, to the CTAs after this one: warp k sends it to
    // ranks q + 1 + k, q + 1 + k + NW, ..., so that the later CTAs get it after
    // one or two stores
    if (rg == 0 && (uint32_t)warp + q + 1 < n) {
        float TA[VEC], TB[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { TA[v] = 1.f; TB[v] = 0.f; }
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float a = sm.a[w2][cq][v];
                TB[v] = __fmaf_rn(a, TB[v], sm.b[w2][cq][v]);
                TA[v] *= a;
            }
#pragma unroll
        for (int i = 0; i < (CL - 1 + NW - 1) / NW; ++i) {  // one pass for clusters of 8, two for 16
            const uint32_t d = q + 1 + (uint32_t)(warp + i * NW);
            if (d >= n) break;
            const uint32_t bar = cluster_map(&cbar, d);
            const uint32_t dst = cluster_map(&cab[q][cq * VEC], d);  // VEC consecutive (A, B) pairs
            if constexpr (VEC == 1) {
                st_async_f2(dst, TA[0], TB[0], bar);
            } else {
#pragma unroll
                for (int v = 0; v < VEC; v += 2)
                    st_async_f4(dst + v * 8, TA[v], TB[v], TA[v + 1], TB[v + 1], bar);
            }
        }
    }
    // the second phase: no CTA leaves while another may still store into it
    // (every store is issued before its CTA arrives; the normal path has also
    // seen every byte land on its barrier before it ends)
    cluster_arrive_relaxed();
    // the warps before this one within the chunk, while the aggregates travel
    float PA[VEC], PB[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { PA[v] = 1.f; PB[v] = 0.f; }
#pragma unroll
    for (int w2 = 0; w2 < NW - 1; ++w2)
        if (w2 < warp)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float a = sm.a[w2][cq][v];
                PB[v] = __fmaf_rn(a, PB[v], sm.b[w2][cq][v]);
                PA[v] *= a;
            }
    {  // every earlier chunk's aggregate is here: a wait of at most cr.spin_limit polls
        bool got = false;
        for (uint32_t k = 0; k <= cr.spin_limit; ++k) {
            if (mbar_try_wait_cluster(&cbar, 0)) {
                got = true;
                break;
            }
            if ((k & 63u) == 63u && (ld_relaxed_u32(cr.err) & ERRBIT_TIMEOUT)) break;
        }
        if (!got) {
            if (lane == 0) atomicOr(cr.err, ERRBIT_TIMEOUT);
#pragma unroll
            for (int v = 0; v < VEC; ++v) s[v] = __int_as_float(0x7fc00000);
        }
    }
#pragma unroll
    for (int d = 0; d < CL - 1; ++d)  // the chunks before this one, in chunk order
        if ((uint32_t)d < q)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float2 e = cab[d][cq * VEC + v];
                s[v] = __fmaf_rn(e.x, s[v], e.y);
            }
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        s[v] = __fmaf_rn(PA[v], s[v], PB[v]);
        s[v] = __fmaf_rn(EA[v], s[v], EB[v]);
    }
    Op::finish(p, g, tc, regs, w, s, xs, acc);
    Op::at_exit(p, xs, acc);
    cluster_wait();
}

// The op's scratch in the TMA strip and segmented kernels: its own space, or
// over the warp aggregates when the op synchronises before using it
// (SCRATCH_IN_CARRY; it keeps the shared memory of two CTAs within an SM).
template <class Op>
using OpScratch = typename std::conditional<Op::SCRATCH_IN_CARRY, int, typename Op::Smem>::type;
template <class Op, class SM>
__device__ __forceinline__ typename Op::Smem& scratch(SM& sm, OpScratch<Op>& own) {
    if constexpr (Op::SCRATCH_IN_CARRY) {
        static_assert(sizeof(typename Op::Smem) <= sizeof(sm.a) + sizeof(sm.b), "op scratch too large");
        return *reinterpret_cast<typename Op::Smem*>(&sm.a[0][0][0]);
    } else {
        return own;
    }
}

// Strip kernel (chain protocol, wide problems): CTA b owns the channel
// strips j = b, b + G, b + 2G, ... (G CTAs) and walks them through time,
// chunk level by chunk level: (0, j1), (0, j2), ..., (1, j1), ...  The state
// after each chunk of a strip stays in this CTA's shared memory, so no tile
// waits for another CTA and nothing is drawn or polled; the tile sequence of
// every CTA is fixed in advance.  Thread 0 keeps ST - 1 tiles of that
// sequence streaming in through the TMA ring: at the top of each iteration,
// after the barrier that also tells it that every warp has copied the
// previous tile into registers, it re-arms that tile's stage with the tile ST
// - 1 ahead.  All warps compute (no producer warp), so two CTAs of 8 warps
// fit an SM with up to 128 registers a thread.
constexpr int STRIP_MAX = 64;  // strips per CTA (state kept in shared memory)

// Use `it` of this CTA: chunk q = it / m of its strip i = it % m, j = b + i*G.
__device__ __forceinline__ void strip_qj(uint32_t G, uint32_t m, uint32_t it, uint32_t& q,
                                         uint32_t& j) {
    q = it / m;
    j = blockIdx.x + (it - q * m) * G;
}

// Thread 0: stage `it % ST` <- the tiles of use `it` (one box per array).
template <class Op, int ST>
__device__ __forceinline__ void strip_issue(const Geom& g, const TmaDesc& td, unsigned char* ring,
                                            uint64_t* full, uint32_t G, uint32_t m, uint32_t it) {
    constexpr int L = Op::NW * Op::R, CW = 32 * Op::VEC;
    constexpr uint32_t SB = tma_stage_bytes<Op>();
    const uint32_t st = it % ST;
    uint32_t q, j;
    strip_qj(G, m, it, q, j);
    const int64_t tchunk = Op::REV ? g.n_chunks - 1 - q : q;
    const int32_t x = (int32_t)(j * CW), y0 = (int32_t)(tchunk * L);
    mbar_arrive_tx(&full[st], td.tx_bytes);
    unsigned char* dst = ring + st * SB;
#pragma unroll
    for (int a = 0; a < Op::TMA_N; ++a)
        if (td.present & (1u << a))
            tma_load_2d(dst + tma_off<Op>(a), &td.map[a], x, y0 + Op::tma_shift(a), &full[st]);
}

// ONEB: one barrier per tile.  The warp aggregates (and an op scratch that
// overlays them) alternate between two buffers by use parity, so a warp may
// start the next tile while another still folds this one; the stop decision
// is read after the carry barrier, and the tile's stage is refilled right
// after it (every warp has copied its tile out by then): two stages keep two
// tiles in flight during the fold and the epilogue.  Otherwise a barrier at
// the top of each tile frees the previous stage.
template <class Op, int ST, bool ONEB>
__global__ void __launch_bounds__(Op::NW * 32, Op::MINB * 8 / Op::NW)
    k_strip(typename Op::Params p, Geom g, uint32_t* err, uint32_t G,
            const __grid_constant__ TmaDesc td) {
    if (Op::skip(p)) return;  // whole launch: before any ticket or barrier
    constexpr int NW = Op::NW, VEC = Op::VEC, L = Op::NW * Op::R;
    constexpr uint32_t SB = tma_stage_bytes<Op>();
    extern __shared__ unsigned char dyn_smem[];
    unsigned char* ring = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + 127) & ~(uintptr_t)127);
    __shared__ StripSmem<VEC, NW> smb[ONEB ? 2 : 1];
    StripSmem<VEC, NW>& sm = smb[0];
    __shared__ OpScratch<Op> xs_own;
    typename Op::Smem& xs = scratch<Op>(sm, xs_own);
    __shared__ __align__(8) uint64_t full[ST];
    __shared__ uint32_t s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // strips of this CTA: j = blockIdx.x + i*G < n_ct; their states (two
    // slots each, by chunk parity) follow the ring
    const uint32_t m = ((uint32_t)g.n_ct - blockIdx.x + G - 1) / G;
    const uint32_t n_it = m * (uint32_t)g.n_chunks;
    float(*carry)[2][32][VEC] = reinterpret_cast<float(*)[2][32][VEC]>(ring + ST * SB);
    uint32_t issued = 0;  // thread 0: uses whose loads were issued
    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) mbar_init(&full[i], 1);
        s_abort = 0;
        mbar_init_fence();
        for (; issued < (uint32_t)ST && issued < n_it; ++issued)
            strip_issue<Op, ST>(g, td, ring, full, G, m, issued);
    }
    __syncthreads();
    typename Op::Acc acc;
    Op::acc_init(acc);
    uint32_t it = 0;
    for (; it < n_it; ++it) {
        const uint32_t st = it % ST;
        if (!mbar_wait(&full[st], (it / ST) & 1u, err)) {
            s_abort = 1;
            atomicOr(err, ERRBIT_TIMEOUT);
        }
        if constexpr (!ONEB) {
            // every warp is done with the previous tile (its stage is free), and
            // the stop decision below is the same in every warp
            csync<NW>();
            if (s_abort != 0) break;
            if (threadIdx.x == 0 && it > 0 && issued < n_it) {
                strip_issue<Op, ST>(g, td, ring, full, G, m, issued);  // into stage (it-1) % ST
                ++issued;
            }
        }
        uint32_t q, j;
        strip_qj(G, m, it, q, j);
        TileCoord tc = tile_coord_qj<Op>(g, q, j);
        tc.acc_run = m == 1;
        tc.acc_flush = m == 1 && (int64_t)q == g.n_chunks - 1;
        typename Op::Regs regs;
        Op::load(SmemSrc<Op>{ring + st * SB, tc.tchunk * L, lane * VEC}, p, g, tc, regs);
        float A[VEC], B[VEC];
        typename Op::Work w;
        Op::aggregate(p, g, tc, regs, w, A, B, true);
        float init[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) init[v] = 0.f;
        const typename Op::S* ip = Op::init_ptr(p);
        if (tc.q == 0 && ip != nullptr && tc.cok) load_vec<typename Op::S, VEC>(ip + tc.c, init);
        float s[VEC];
        if constexpr (ONEB) {
            const int pb = (int)(it & 1u);
            StripSmem<VEC, NW>& sb = smb[pb];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                sb.a[warp][lane][v] = A[v];
                sb.b[warp][lane][v] = B[v];
            }
            csync<NW>();  // the tile's one barrier
            if (s_abort != 0) break;
            if (threadIdx.x == 0 && issued < n_it) {
                strip_issue<Op, ST>(g, td, ring, full, G, m, issued);  // into stage st
                ++issued;
            }
            float(*cs)[32][VEC] = carry[it % m];
            const int par = (int)(q & 1u);
            float stt[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v)
                stt[v] = tc.q == 0 ? (tc.cok ? init[v] : 0.f) : cs[par][lane][v];
#pragma unroll kFoldUnroll
            for (int w2 = 0; w2 < warp; ++w2)
#pragma unroll
                for (int v = 0; v < VEC; ++v) stt[v] = __fmaf_rn(sb.a[w2][lane][v], stt[v], sb.b[w2][lane][v]);
            if (warp == NW - 1) {
#pragma unroll
                for (int v = 0; v < VEC; ++v) cs[par ^ 1][lane][v] = __fmaf_rn(A[v], stt[v], B[v]);
            }
#pragma unroll
            for (int v = 0; v < VEC; ++v) s[v] = stt[v];
            Op::finish(p, g, tc, regs, w, s, scratch<Op>(sb, xs_own), acc);
        } else {
            strip_carry<VEC, NW>(sm, A, B, init, s, carry[it % m], (int)(q & 1u), tc.q == 0, tc.cok);
            Op::finish(p, g, tc, regs, w, s, xs, acc);
        }
    }
    Op::at_exit(p, xs, acc);
    if (threadIdx.x == 0)  // after an early stop: copies still in flight land first
        for (uint32_t i = it; i < issued; ++i) mbar_wait(&full[i % ST], (i / ST) & 1u, err);
}

// Segmented walker kernel (walker protocol, TMA staging; long, narrow
// problems).  The unit of work (ticket) is a segment: SEG consecutive chunks
// of one channel strip, streamed through the TMA ring twice.  At its own
// iteration i a CTA
//   1. reduces the segment of its ticket i (from HBM, kept in L2): folds the
//      chunk aggregates into the segment's aggregate and publishes it;
//   2. consumes the segment of its ticket i-SEG_LAG (from L2): one wait for
//      the state entering that segment, which the walker CTAs (the first
//      tickets) fold from the segment aggregates, then the state is carried
//      from chunk to chunk in shared memory, as in the strip kernel, and the
//      outputs are written.
// A reduce-only launch (NextAgg::reduce_only) has no walkers and no consume
// pass: its reduce pass publishes the segment aggregates into NextAgg::agg
// with the next launch's epoch -- the aggregates of a DEER solve's first
// iteration, which then runs consume-only like the later ones.
// The lag of SEG_LAG segments gives the walkers that many segments' time to
// produce every entering state, while SEG_LAG + 1 short segments per CTA stay
// within the L2.  Tickets, aggregate packets, walker work and the carry wait
// are paid once per segment rather than once per tile, and every load is
// issued ST - 1 uses ahead by thread 0 (tickets are drawn one iteration
// early).  A consume only waits for reduces of smaller tickets, and every CTA
// reduces before it consumes: every wait ends.
//
// Operations whose next launch's coefficients are built from this launch's
// outputs (DEER: iteration k+1's Jacobian and right-hand side at row t come
// from y^(k)_{t-1} and u_t) also fold, in the consume pass, the segment
// aggregates of the next launch and publish them with its epoch
// (NEXT_AGG, NextAgg::agg).  A launch whose aggregates were published that way
// (NextAgg::pre) has no reduce pass: each ticket is consumed at once, its
// tiles read from HBM once, while the walkers fold aggregates that are all
// visible from the start.
#ifndef LR_SEG_LAG
#define LR_SEG_LAG 2
#endif
constexpr int SEG_LAG = LR_SEG_LAG;  // iterations between a segment's two passes

struct SegGeom {
    uint32_t seg;      // chunks per segment
    uint32_t n_seg;    // segments per strip: ceil(n_chunks / seg)
    uint32_t n_units;  // n_seg * n_ct
};

// The next launch's segment aggregates, and nothing else (the pass before a
// DEER solve's first iteration, whose aggregates depend on the inputs only):
// a plain streaming reduction.  CTA b takes segments (units) b, b + G, ...; in
// a segment warp w folds the rows of its contiguous share [w S/NW, (w+1) S/NW)
// (S rows per segment) from global memory, R rows per step and two steps in
// flight, and warp 0 folds the NW shares in row order and publishes the
// segment's packets with the next launch's epoch.  Nothing waits: every CTA
// draws one ticket only to learn the launch's epoch and to retire it.  The
// association is fixed by position (rows of a step in order, steps in order,
// then the warps' shares in order).
template <class Op>
__global__ void __launch_bounds__(Op::NW * 32, Op::MINB * 8 / Op::NW)
    k_segred(typename Op::Params p, Geom g, const Carry cr0, SegGeom sg) {
    static_assert(has_next_agg<Op>::value, "a reduce-only launch publishes the next aggregates");
    if (Op::skip(p)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) retire_epoch(cr0);
        return;
    }
    constexpr int NW = Op::NW, VEC = Op::VEC, R = Op::R, L = NW * R, CW = 32 * VEC;
    __shared__ float sa[NW][32][VEC], sb[NW][32][VEC];
    __shared__ uint32_t s_epoch;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Carry cr = cr0;
    NextAgg nx = Op::next_agg(p);
    if (threadIdx.x == 0) {
        const uint32_t t = draw_ticket(cr);
        ticket_drawn(cr, g, t);
        s_epoch = cr.epoch;
    }
    __syncthreads();
    nx.epoch = epoch_after(s_epoch);  // the next launch's
    const uint64_t pol = l2_evict_first();  // every row is read once
    const int64_t seg_rows = (int64_t)sg.seg * L, share = seg_rows / NW;
    for (uint32_t unit = blockIdx.x; unit < sg.n_units; unit += gridDim.x) {
        const uint32_t seg = unit / (uint32_t)g.n_ct, j = unit - seg * (uint32_t)g.n_ct;
        TileCoord tc;
        tc.c = (int64_t)j * CW + lane * VEC;
        tc.cd = chan_feat(g, tc.c);
        tc.cok = tc.c < g.C;
        tc.acc_run = false;
        tc.acc_flush = false;
        const int64_t r0 = (int64_t)seg * seg_rows + warp * share;
        float WA[VEC], WB[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { WA[v] = 1.f; WB[v] = 0.f; }
        const GlobalSrcHint src{g.C, tc.c, pol};
        for (int64_t k = 0; k < share; k += 2 * R) {
            typename Op::Regs rg[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                tc.t0 = r0 + k + h * R;
                tc.q = tc.t0 / L;
                tc.tchunk = tc.q;
                if (k + h * R < share && tc.t0 < g.T) Op::load(src, p, g, tc, rg[h]);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                tc.t0 = r0 + k + h * R;
                tc.q = tc.t0 / L;
                tc.tchunk = tc.q;
                if (k + h * R < share && tc.t0 < g.T) {
                    typename Op::Work w;
                    float A[VEC], B[VEC];
                    Op::aggregate(p, g, tc, rg[h], w, A, B, false);
#pragma unroll
                    for (int v = 0; v < VEC; ++v) {
                        WB[v] = __fmaf_rn(A[v], WB[v], B[v]);
                        WA[v] *= A[v];
                    }
                }
            }
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            sa[warp][lane][v] = WA[v];
            sb[warp][lane][v] = WB[v];
        }
        __syncthreads();
        if (warp == 0 && tc.cok && seg + 1 < sg.n_seg) {
            float SA[VEC], SBv[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) { SA[v] = 1.f; SBv[v] = 0.f; }
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2)
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    const float a = sa[w2][lane][v];
                    SBv[v] = __fmaf_rn(a, SBv[v], sb[w2][lane][v]);
                    SA[v] *= a;
                }
#pragma unroll
            for (int v = 0; v < VEC; ++v)
                st_pkt2(nx.agg + 2 * ((tc.c + v) * sg.n_seg + seg), pkt(SA[v], nx.epoch),
                        pkt(SBv[v], nx.epoch));
        }
        __syncthreads();  // sa / sb are rewritten by the next segment
    }
}

template <class Op, int ST>
__device__ __forceinline__ void seg_issue(const Geom& g, const TmaDesc& td, unsigned char* ring,
                                          uint64_t* full, uint32_t st, uint32_t q, uint32_t j,
                                          uint64_t pol) {
    constexpr int L = Op::NW * Op::R, CW = 32 * Op::VEC;
    const int64_t tchunk = Op::REV ? g.n_chunks - 1 - (int64_t)q : (int64_t)q;
    const int32_t x = (int32_t)((int64_t)j * CW), y0 = (int32_t)(tchunk * L);
    mbar_arrive_tx(&full[st], td.tx_bytes);
    unsigned char* dst = ring + st * tma_stage_bytes<Op>();
#pragma unroll
    for (int a = 0; a < Op::TMA_N; ++a)
        if (td.present & (1u << a))
            tma_load_2d_hint(dst + tma_off<Op>(a), &td.map[a], x, y0 + Op::tma_shift(a), &full[st],
                             pol);
}

// Per-warp partials of the next launch's aggregate of the chunk just
// finished (k_seg, NEXT_AGG operations).  They live in that chunk's ring
// stage: its tile is in registers by then, and the stage is refilled only
// after the next barrier, once warp 0 has folded them.
template <int VEC, int NW>
struct NextPart {
    float a[NW][32][VEC];
    float b[NW][32][VEC];
};

template <class Op, int ST>
__global__ void __launch_bounds__(Op::NW * 32, Op::MINB * 8 / Op::NW)
    k_seg(typename Op::Params p, Geom g, const Carry cr0, SegGeom sg,
          const __grid_constant__ TmaDesc td) {
    if (Op::skip(p)) {  // whole launch: before any ticket or barrier
        if (blockIdx.x == 0 && threadIdx.x == 0) retire_epoch(cr0);
        return;
    }
    Carry cr = cr0;
    constexpr int NW = Op::NW, VEC = Op::VEC, L = Op::NW * Op::R;
    constexpr uint32_t SB = tma_stage_bytes<Op>();
    constexpr bool NXT = has_next_agg<Op>::value;
    extern __shared__ unsigned char dyn_smem[];
    unsigned char* ring = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + 127) & ~(uintptr_t)127);
    __shared__ StripSmem<VEC, NW> sm;
    __shared__ OpScratch<Op> xs_own;
    typename Op::Smem& xs = scratch<Op>(sm, xs_own);
    __shared__ float carry[2][32][VEC];  // by chunk parity
    __shared__ __align__(8) uint64_t full[ST];
    __shared__ uint32_t s_tk[2], s_abort, s_epoch;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    NextAgg nx{nullptr, 0u, 0u, 0u};
    if constexpr (NXT) nx = Op::next_agg(p);
    const bool pre = nx.pre != 0;
    const bool ronly = NXT && nx.reduce_only != 0;
    if (ronly) cr.n_walk = 0;  // no walkers: nothing is consumed
    const uint32_t limit = cr.n_walk + sg.n_units;
    static_assert(!NXT || sizeof(NextPart<VEC, NW>) <= SB, "partials must fit in a stage");
    // uses per iteration: the reduce pass (none when pre), the consume pass
    // (none when reduce-only)
    const uint32_t nred = pre ? 0u : sg.seg;
    const uint32_t uses = nred + (ronly ? 0u : sg.seg);
    if (threadIdx.x == 0) {
        const uint32_t t = draw_ticket(cr);
        ticket_drawn(cr, g, t);
        s_tk[0] = t;
        s_abort = 0;
        s_epoch = cr.epoch;
    }
    __syncthreads();
    cr.epoch = s_epoch;
    nx.epoch = epoch_after(cr.epoch);  // the next launch's
    uint32_t cur = s_tk[0];
    if (cur < cr.n_walk) {  // walker role: its chunks are the segments
        Geom gw = g;
        gw.n_chunks = sg.n_seg;
        walker<typename Op::S, NW>(cr, gw, cur, Op::init_ptr(p));
        return;
    }
    if (cur >= limit) return;
    // thread 0 state: tickets drawn ahead, loads issued ahead
    bool drawing = true;
    uint32_t pend = 0;
    uint32_t inflight = 0;  // stages with a box in flight
    uint64_t pol_keep = 0, pol_drop = 0;
    // Thread 0: issue use u into stage u % ST.  Use u is chunk k of the reduce
    // pass of ticket `red` (k < nred) or chunk k - nred of the consume pass of
    // ticket `con`; tickets >= limit have no segment.
    auto issue = [&](uint32_t u, uint32_t red, uint32_t con) {
        const uint32_t k = u % uses;
        const uint32_t tk = k < nred ? red : con, c = k < nred ? k : k - nred;
        if (tk >= limit) return;
        const uint32_t x = tk - cr.n_walk, seg = x / (uint32_t)g.n_ct;
        const uint32_t j = x - seg * (uint32_t)g.n_ct, q = seg * sg.seg + c;
        if (q >= (uint32_t)g.n_chunks) return;
        const uint32_t st = u % ST;
        seg_issue<Op, ST>(g, td, ring, full, st, q, j, k < nred ? pol_keep : pol_drop);
        inflight |= 1u << st;
    };
    // tq[0]: ticket consumed this iteration, tq[SEG_LAG]: reduced this
    // iteration, tq[SEG_LAG + 1]: reduced next iteration.  Without a reduce
    // pass (pre) tq[SEG_LAG] is consumed this iteration and tq[SEG_LAG + 1]
    // the next.
    uint32_t tq[SEG_LAG + 2];
#pragma unroll
    for (int i = 0; i < SEG_LAG; ++i) tq[i] = limit;
    tq[SEG_LAG] = cur;
    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) mbar_init(&full[i], 1);
        mbar_init_fence();
        pol_keep = l2_evict_last();
        pol_drop = l2_evict_first();
        const uint32_t t1 = draw_ticket(cr);
        ticket_drawn(cr, g, t1);
        if (t1 >= limit) drawing = false;
        s_tk[1] = t1;
        // uses 0 .. ST-1: the first chunks of the reduce pass of `cur`, or of
        // its consume pass when pre (the launch keeps SEG >= ST)
        for (uint32_t u = 0; u < (uint32_t)ST; ++u) issue(u, cur, pre ? cur : limit);
        if (drawing) pend = draw_ticket(cr);
    }
    __syncthreads();
    tq[SEG_LAG + 1] = s_tk[1];
    uint32_t phase = 0;  // parity of the next completion of each stage's barrier
    uint32_t it = 0;     // uses consumed
    typename Op::Acc acc;
    Op::acc_init(acc);
    bool stop = false;
    // Next launch's aggregate of the segment being consumed: warp 0 folds the
    // chunks' warp partials (written into a chunk's stage after its finish,
    // read after the next barrier, before that stage is refilled) in row order.
    float NA[VEC], NB[VEC];
    bool nx_pend = false;  // partials of the previous chunk await the fold
    uint32_t nx_st = 0;    // the stage holding them
    auto nx_fold = [&]() {
        if constexpr (NXT) {
            if (warp == 0 && nx_pend) {
                const NextPart<VEC, NW>& np =
                    *reinterpret_cast<const NextPart<VEC, NW>*>(ring + nx_st * SB);
#pragma unroll
                for (int w2 = 0; w2 < NW; ++w2)
#pragma unroll
                    for (int v = 0; v < VEC; ++v) {
                        const float a = np.a[w2][lane][v];
                        NB[v] = __fmaf_rn(a, NB[v], np.b[w2][lane][v]);
                        NA[v] *= a;
                    }
                __syncwarp();  // every lane has read them before thread 0 refills the stage
            }
        }
        nx_pend = false;
    };
    // Top of use `it`: wait for its box, then a barrier after which the stage
    // of use it-1 is free and the stop decision is uniform; refill that stage
    // with use it-1+ST (this iteration's tickets, or the next iteration's).
    auto top = [&](bool valid) {
        const uint32_t st = it % ST;
        if (valid && !mbar_wait(&full[st], (phase >> st) & 1u, cr.err)) s_abort = 1;
        csync<NW>();
        if (s_abort != 0) return false;
        nx_fold();  // the previous chunk's partials, in the stage refilled next
        if (threadIdx.x == 0 && it > 0) {
            const uint32_t u = it - 1 + ST;
            if (u / uses == it / uses) issue(u, tq[SEG_LAG], pre ? tq[SEG_LAG] : tq[0]);
            else issue(u, tq[SEG_LAG + 1], pre ? tq[SEG_LAG + 1] : tq[1]);
        }
        if (valid) {
            phase ^= 1u << st;
            if (threadIdx.x == 0) inflight &= ~(1u << st);
        }
        return true;
    };
    auto active = [&]() {
        bool a = tq[SEG_LAG] < limit;
#pragma unroll
        for (int i = 0; i < SEG_LAG; ++i) a = a || (!pre && !ronly && tq[i] < limit);
        return a;
    };
    while (active() && !stop) {
        const uint32_t tk_red = pre ? limit : tq[SEG_LAG], tk_con = pre ? tq[SEG_LAG] : tq[0];
        // ---- pass 1: the aggregate of the segment of `tk_red`
        const bool has_red = tk_red < limit;
        const uint32_t xr = has_red ? tk_red - cr.n_walk : 0u;
        const uint32_t seg_r = xr / (uint32_t)g.n_ct, j_r = xr - seg_r * (uint32_t)g.n_ct;
        float SA[VEC], SBv[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { SA[v] = 1.f; SBv[v] = 0.f; }
        for (uint32_t c = 0; c < nred; ++c, ++it) {
            const uint32_t q = seg_r * sg.seg + c;
            const bool valid = has_red && q < (uint32_t)g.n_chunks;
            if (!top(valid)) { stop = true; break; }
            if (!valid) continue;
            const TileCoord tc = tile_coord_qj<Op>(g, q, j_r);
            typename Op::Regs regs;
            typename Op::Work w;
            Op::load(SmemSrc<Op>{ring + (it % ST) * SB, tc.tchunk * L, lane * VEC}, p, g, tc, regs);
            float A[VEC], B[VEC];
            Op::aggregate(p, g, tc, regs, w, A, B, false);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                sm.a[warp][lane][v] = A[v];
                sm.b[warp][lane][v] = B[v];
            }
            csync<NW>();
            if (warp == 0) {  // fold the warps (row order), then into the segment
#pragma unroll
                for (int w2 = 0; w2 < NW; ++w2)
#pragma unroll
                    for (int v = 0; v < VEC; ++v) {
                        const float a = sm.a[w2][lane][v];
                        SBv[v] = __fmaf_rn(a, SBv[v], sm.b[w2][lane][v]);
                        SA[v] *= a;
                    }
            }
        }
        if (stop) break;
        if (warp == 0 && has_red) {  // the segment's aggregate, for the walkers (or the next launch's)
            const TileCoord tc = tile_coord_qj<Op>(g, seg_r * sg.seg, j_r);
            u64* dst = ronly ? nx.agg : cr.agg;
            const uint32_t ep = ronly ? nx.epoch : cr.epoch;
            if (tc.cok && seg_r + 1 < sg.n_seg) {
#pragma unroll
                for (int v = 0; v < VEC; ++v)
                    st_pkt2(dst + 2 * ((tc.c + v) * sg.n_seg + seg_r), pkt(SA[v], ep), pkt(SBv[v], ep));
            }
        }
        // ---- pass 2: the outputs of the segment of `tk_con`
        const bool has_con = !ronly && tk_con < limit;
        const uint32_t xc = has_con ? tk_con - cr.n_walk : 0u;
        const uint32_t seg_c = xc / (uint32_t)g.n_ct, j_c = xc - seg_c * (uint32_t)g.n_ct;
        if (warp == 0 && has_con) {  // the state entering that segment
            const TileCoord tc = tile_coord_qj<Op>(g, seg_c * sg.seg, j_c);
            float cin[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) cin[v] = 0.f;
            const typename Op::S* ip = Op::init_ptr(p);
            if (seg_c == 0) {
                if (tc.cok && ip != nullptr) load_vec<typename Op::S, VEC>(ip + tc.c, cin);
            } else {
                uint32_t spins = 0, sleep_ns = 0;
                while (true) {
                    const bool ok = !tc.cok || get_states_strided<VEC>(
                                                   cr.inc + tc.c * sg.n_seg + seg_c - 1, sg.n_seg,
                                                   cin, cr.epoch);
                    if (__all_sync(0xffffffffu, ok)) break;
                    if (__any_sync(0xffffffffu, wait_step(cr, spins, sleep_ns, kTileMaxSleepNs))) {
                        if (lane == 0) give_up(cr);
#pragma unroll
                        for (int v = 0; v < VEC; ++v) cin[v] = __int_as_float(0x7fc00000);
                        break;
                    }
                }
            }
#pragma unroll
            for (int v = 0; v < VEC; ++v) carry[0][lane][v] = cin[v];
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) { NA[v] = 1.f; NB[v] = 0.f; }
        for (uint32_t c = 0; c < (ronly ? 0u : sg.seg); ++c, ++it) {
            const uint32_t q = seg_c * sg.seg + c;
            const bool valid = has_con && q < (uint32_t)g.n_chunks;
            if (!top(valid)) { stop = true; break; }
            if (!valid) continue;
            TileCoord tc = tile_coord_qj<Op>(g, q, j_c);
            tc.acc_run = true;  // the segment's chunks, in scan order
            tc.acc_flush = c + 1 == sg.seg || (int64_t)q + 1 == g.n_chunks;
            typename Op::Regs regs;
            typename Op::Work w;
            Op::load(SmemSrc<Op>{ring + (it % ST) * SB, tc.tchunk * L, lane * VEC}, p, g, tc, regs);
            float A[VEC], B[VEC];
            Op::aggregate(p, g, tc, regs, w, A, B, true);
            float s0[VEC], st[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) s0[v] = 0.f;
            strip_carry<VEC, NW>(sm, A, B, s0, st, carry, (int)(c & 1u), false, tc.cok);
            Op::finish(p, g, tc, regs, w, st, xs, acc);
            if constexpr (NXT) {
                if (nx.agg != nullptr) {
                    // into this chunk's stage: every warp copied its tile out
                    // of it before the barrier inside strip_carry
                    NextPart<VEC, NW>& np = *reinterpret_cast<NextPart<VEC, NW>*>(ring + (it % ST) * SB);
#pragma unroll
                    for (int v = 0; v < VEC; ++v) {
                        np.a[warp][lane][v] = w.NA[v];
                        np.b[warp][lane][v] = w.NB[v];
                    }
                    fence_proxy_async_smem();  // ordered before the copy that refills the stage
                    nx_pend = true;
                    nx_st = it % ST;
                }
            }
        }
        if (stop) break;
        if constexpr (NXT) {
            if (nx.agg != nullptr && has_con) {
                csync<NW>();
                nx_fold();
                const TileCoord tc = tile_coord_qj<Op>(g, seg_c * sg.seg, j_c);
                if (warp == 0 && tc.cok && seg_c + 1 < sg.n_seg) {
#pragma unroll
                    for (int v = 0; v < VEC; ++v)
                        st_pkt2(nx.agg + 2 * ((tc.c + v) * sg.n_seg + seg_c), pkt(NA[v], nx.epoch),
                                pkt(NB[v], nx.epoch));
                }
                // the ticket step below ends with a block barrier before any
                // warp writes partials again
            }
        }
        // ---- next iteration: shift the ticket queue, append the one drawn
        if (threadIdx.x == 0) {
            uint32_t t2 = limit;
            if (drawing) {
                t2 = pend;
                ticket_drawn(cr, g, t2);
                if (t2 >= limit) drawing = false;
                else pend = draw_ticket(cr);
            }
            s_tk[0] = t2;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i <= SEG_LAG; ++i) tq[i] = tq[i + 1];
        tq[SEG_LAG + 1] = s_tk[0];
    }
    if (stop && threadIdx.x == 0) give_up(cr);
    Op::at_exit(p, xs, acc);
    if (threadIdx.x == 0)  // after an early stop: boxes still in flight land first
        for (int st = 0; st < ST; ++st)
            if (inflight & (1u << st)) mbar_wait(&full[st], (phase >> st) & 1u, cr.err);
}

// Segmented walker kernel, consume only: a launch whose segment aggregates
// the previous launch published (NEXT_AGG operations with NextAgg::pre: DEER
// iterations after the first).  Each ticket (segment) is consumed as soon as
// it is drawn, its tiles read from HBM once.  One barrier per chunk: the warp
// aggregates and the next launch's per-warp partials alternate between two
// buffers by chunk parity (a warp may start the next chunk while another is
// still folding this one), the stop decision is read after that barrier, and
// a chunk's stage is refilled right after it -- every warp has copied its tile
// out by then -- so two stages keep two tiles in flight during the fold and
// the epilogue.
template <class Op, int ST>
__global__ void __launch_bounds__(Op::NW * 32, Op::MINB * 8 / Op::NW)
    k_seg1(typename Op::Params p, Geom g, const Carry cr0, SegGeom sg,
           const __grid_constant__ TmaDesc td) {
    static_assert(has_next_agg<Op>::value, "a consume-only launch publishes the next aggregates");
    if (Op::skip(p)) {  // whole launch: before any ticket or barrier
        if (blockIdx.x == 0 && threadIdx.x == 0) retire_epoch(cr0);
        return;
    }
    Carry cr = cr0;
    constexpr int NW = Op::NW, VEC = Op::VEC, L = Op::NW * Op::R;
    constexpr uint32_t SB = tma_stage_bytes<Op>();
    extern __shared__ unsigned char dyn_smem[];
    unsigned char* ring = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + 127) & ~(uintptr_t)127);
    __shared__ StripSmem<VEC, NW> sm[2];
    __shared__ NextPart<VEC, NW> part[2];
    __shared__ typename Op::Smem xs;
    __shared__ float carry[2][32][VEC];  // by chunk parity
    __shared__ __align__(8) uint64_t full[ST];
    __shared__ uint32_t s_tk[2], s_abort, s_epoch;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t limit = cr.n_walk + sg.n_units;
    NextAgg nx = Op::next_agg(p);
    if (threadIdx.x == 0) {
        const uint32_t t = draw_ticket(cr);
        ticket_drawn(cr, g, t);
        s_tk[0] = t;
        s_abort = 0;
        s_epoch = cr.epoch;
    }
    __syncthreads();
    cr.epoch = s_epoch;
    nx.epoch = epoch_after(cr.epoch);  // the next launch's
    const uint32_t cur = s_tk[0];
    if (cur < cr.n_walk) {  // walker role: its chunks are the segments
        Geom gw = g;
        gw.n_chunks = sg.n_seg;
        walker<typename Op::S, NW>(cr, gw, cur, Op::init_ptr(p));
        return;
    }
    if (cur >= limit) return;
    // thread 0 state: the ticket drawn ahead, loads issued ahead
    bool drawing = true;
    uint32_t pend = 0;
    uint32_t inflight = 0;  // stages with a box in flight
    uint64_t pol = 0;
    uint32_t tk = cur, tk_next = limit;
    // Thread 0: issue use u (chunk u % SEG of the ticket whose uses it is
    // part of: every ticket has SEG uses) into stage u % ST.
    auto issue = [&](uint32_t u, uint32_t t) {
        if (t >= limit) return;
        const uint32_t x = t - cr.n_walk, seg = x / (uint32_t)g.n_ct;
        const uint32_t j = x - seg * (uint32_t)g.n_ct, q = seg * sg.seg + u % sg.seg;
        if (q >= (uint32_t)g.n_chunks) return;
        const uint32_t st = u % ST;
        seg_issue<Op, ST>(g, td, ring, full, st, q, j, pol);
        inflight |= 1u << st;
    };
    // Thread 0, once use u's stage is free: issue use u + ST (the same
    // ticket's, or the next one's; SEG >= ST).
    auto refill = [&](uint32_t u) {
        if (threadIdx.x == 0) {
            const uint32_t v = u + ST;
            issue(v, v / sg.seg == u / sg.seg ? tk : tk_next);
        }
    };
    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) mbar_init(&full[i], 1);
        mbar_init_fence();
        pol = l2_evict_first();  // every tile is read once
        const uint32_t t1 = draw_ticket(cr);
        ticket_drawn(cr, g, t1);
        if (t1 >= limit) drawing = false;
        s_tk[1] = t1;
        tk_next = t1;
        for (uint32_t u = 0; u < (uint32_t)ST; ++u) issue(u, cur);
        if (drawing) pend = draw_ticket(cr);
    }
    __syncthreads();
    tk_next = s_tk[1];
    uint32_t phase = 0;  // parity of the next completion of each stage's barrier
    uint32_t it = 0;     // uses consumed
    typename Op::Acc acc;
    Op::acc_init(acc);
    bool stop = false;
    while (tk < limit) {
        const uint32_t x = tk - cr.n_walk;
        const uint32_t seg_c = x / (uint32_t)g.n_ct, j_c = x - seg_c * (uint32_t)g.n_ct;
        if (warp == 0) {  // the state entering the segment, from the walkers
            const TileCoord tc = tile_coord_qj<Op>(g, seg_c * sg.seg, j_c);
            float cin[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) cin[v] = 0.f;
            const typename Op::S* ip = Op::init_ptr(p);
            if (seg_c == 0) {
                if (tc.cok && ip != nullptr) load_vec<typename Op::S, VEC>(ip + tc.c, cin);
            } else {
                uint32_t spins = 0, sleep_ns = 0;
                while (true) {
                    const bool ok = !tc.cok || get_states_strided<VEC>(
                                                   cr.inc + tc.c * sg.n_seg + seg_c - 1, sg.n_seg,
                                                   cin, cr.epoch);
                    if (__all_sync(0xffffffffu, ok)) break;
                    if (__any_sync(0xffffffffu, wait_step(cr, spins, sleep_ns, kTileMaxSleepNs))) {
                        if (lane == 0) give_up(cr);
#pragma unroll
                        for (int v = 0; v < VEC; ++v) cin[v] = __int_as_float(0x7fc00000);
                        break;
                    }
                }
            }
#pragma unroll
            for (int v = 0; v < VEC; ++v) carry[0][lane][v] = cin[v];
        }
        float NA[VEC], NB[VEC];  // warp 0: the next launch's aggregate of this segment
#pragma unroll
        for (int v = 0; v < VEC; ++v) { NA[v] = 1.f; NB[v] = 0.f; }
        int pend_buf = -1;  // part[] buffer whose partials await warp 0's fold
        auto fold_part = [&]() {
            if (warp == 0 && pend_buf >= 0) {
#pragma unroll
                for (int w2 = 0; w2 < NW; ++w2)
#pragma unroll
                    for (int v = 0; v < VEC; ++v) {
                        const float a = part[pend_buf].a[w2][lane][v];
                        NB[v] = __fmaf_rn(a, NB[v], part[pend_buf].b[w2][lane][v]);
                        NA[v] *= a;
                    }
            }
            pend_buf = -1;
        };
        for (uint32_t c = 0; c < sg.seg; ++c, ++it) {
            const uint32_t q = seg_c * sg.seg + c;
            const uint32_t st = it % ST;
            if (q >= (uint32_t)g.n_chunks) {  // past the strip's end: no box, stage idle
                refill(it);
                continue;
            }
            if (!mbar_wait(&full[st], (phase >> st) & 1u, cr.err)) s_abort = 1;
            phase ^= 1u << st;
            const TileCoord tc = tile_coord_qj<Op>(g, q, j_c);
            typename Op::Regs regs;
            typename Op::Work w;
            Op::load(SmemSrc<Op>{ring + st * SB, tc.tchunk * L, lane * VEC}, p, g, tc, regs);
            float A[VEC], B[VEC];
            Op::aggregate(p, g, tc, regs, w, A, B, true);
            const int par = (int)(c & 1u);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                sm[par].a[warp][lane][v] = A[v];
                sm[par].b[warp][lane][v] = B[v];
            }
            csync<NW>();  // the chunk's one barrier
            if (s_abort != 0) { stop = true; break; }
            if (threadIdx.x == 0) inflight &= ~(1u << st);
            refill(it);  // every warp has copied its tile out of stage st
            fold_part();  // the previous chunk's partials
            float s0[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) s0[v] = carry[par][lane][v];
#pragma unroll kFoldUnroll
            for (int w2 = 0; w2 < warp; ++w2)
#pragma unroll
                for (int v = 0; v < VEC; ++v)
                    s0[v] = __fmaf_rn(sm[par].a[w2][lane][v], s0[v], sm[par].b[w2][lane][v]);
            if (warp == NW - 1) {
#pragma unroll
                for (int v = 0; v < VEC; ++v) carry[par ^ 1][lane][v] = __fmaf_rn(A[v], s0[v], B[v]);
            }
            Op::finish(p, g, tc, regs, w, s0, xs, acc);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                part[par].a[warp][lane][v] = w.NA[v];
                part[par].b[warp][lane][v] = w.NB[v];
            }
            pend_buf = par;
        }
        if (stop) break;
        csync<NW>();  // the last chunk's partials are visible
        fold_part();
        {
            const TileCoord tc = tile_coord_qj<Op>(g, seg_c * sg.seg, j_c);
            if (warp == 0 && tc.cok && seg_c + 1 < sg.n_seg) {
#pragma unroll
                for (int v = 0; v < VEC; ++v)
                    st_pkt2(nx.agg + 2 * ((tc.c + v) * sg.n_seg + seg_c), pkt(NA[v], nx.epoch),
                            pkt(NB[v], nx.epoch));
            }
        }
        // next ticket (drawn one ahead)
        if (threadIdx.x == 0) {
            uint32_t t2 = limit;
            if (drawing) {
                t2 = pend;
                ticket_drawn(cr, g, t2);
                if (t2 >= limit) drawing = false;
                else pend = draw_ticket(cr);
            }
            s_tk[0] = t2;
        }
        __syncthreads();  // also: no warp writes sm / part / carry of the next segment early
        tk = tk_next;
        tk_next = s_tk[0];
    }
    if (stop && threadIdx.x == 0) give_up(cr);
    Op::at_exit(p, xs, acc);
    if (threadIdx.x == 0)  // after an early stop: boxes still in flight land first
        for (int st = 0; st < ST; ++st)
            if (inflight & (1u << st)) mbar_wait(&full[st], (phase >> st) & 1u, cr.err);
}

template <class Op>
int chain_occupancy() {
    static int occ[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& o = occ[dev & 63];
    if (o <= 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_chain<Op>, 32 * Op::NW, 0) !=
                cudaSuccess ||
            n <= 0)
            n = 1;
        o = n;
    }
    return o;
}

// Resident CTAs of k_stream<Op> per SM (cached per device).
template <class Op>
int stream_occupancy() {
    static int occ[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& o = occ[dev & 63];
    if (o <= 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_stream<Op>, 32 * Op::NW, 0) !=
                cudaSuccess ||
            n <= 0)
            n = 1;
        o = n;
    }
    return o;
}

// Host: launch k_chain<Op> (chain protocol).  The register double buffer
// hides the load latency.
template <class Op>
cudaError_t launch_chain(const typename Op::Params& p, Geom g, const Carry& cr, cudaStream_t s) {
    const uint32_t grid = persist_grid(g, cr, chain_occupancy<Op>());
    g.n_draws = g.n_tiles + grid - g.ticket_base;
    k_chain<Op><<<grid, 32 * Op::NW, 0, s>>>(p, g, cr);
    return cudaGetLastError();
}

// Host: launch k_stream<Op> (walker protocol).  The consume lag d_con is
// LR_STREAM_LAG rounds of tickets (one ticket per tile CTA; two rounds
// measured best on GB300), capped so that the tiles in flight (about 32 MB of
// inputs) stay well within the L2.
template <class Op>
cudaError_t launch_wstream(const typename Op::Params& p, Geom g, Carry cr, cudaStream_t s);
template <class Op>
cudaError_t launch_stream(const typename Op::Params& p, Geom g, const Carry& cr, cudaStream_t s) {
    if constexpr (stream_ws<Op>::value) {
        const cudaError_t e = launch_wstream<Op>(p, g, cr, s);
        if (e != cudaErrorNotSupported) return e;
    }
    const uint32_t grid = persist_grid(g, cr, stream_occupancy<Op>());
    const uint64_t tile_ctas = grid > cr.n_walk ? grid - cr.n_walk : 1;
    const uint64_t tile_bytes =
        (uint64_t)Op::NW * Op::R * 32 * Op::VEC * sizeof(typename Op::S) * Op::IN_ARRAYS;
    uint64_t d_con = LR_STREAM_LAG * tile_ctas;
    const uint64_t cap = ((uint64_t)LR_STREAM_L2MB << 20) / (tile_bytes ? tile_bytes : 1);
    if (d_con > cap) d_con = cap > 1 ? cap : 1;
    g.n_draws = g.n_tiles + (uint32_t)d_con + grid - g.ticket_base;
    k_stream<Op><<<grid, 32 * Op::NW, 0, s>>>(p, g, cr, (uint32_t)d_con);
    return cudaGetLastError();
}

// Host: launch k_wstream<Op> (walker protocol, warp-specialised, TMA).
// cudaErrorNotSupported when it does not apply (the walker warps would
// outnumber the CTAs, or the arrays cannot be tensor-mapped).
template <class Op>
cudaError_t launch_wstream(const typename Op::Params& p, Geom g, Carry cr, cudaStream_t s) {
    using Ly = WsLayout<Op>;
    constexpr int CW = 32 * Op::VEC;
    constexpr uint32_t SB = Ly::SB;
    constexpr size_t dyn = (size_t)(Ly::STR + Ly::STC) * SB + 128;
    static_assert(Op::TMA_N <= TMA_MAX_ARR, "too many staged arrays");
    static_assert(Ly::SR + 1 <= 256 && CW <= 256, "a TMA box holds at most 256 rows and columns");
    if (Op::VEC != 4 || cr.wv <= 0) return cudaErrorNotSupported;
    TmaDesc td;
    memset(&td, 0, sizeof td);
    const void* ptr[TMA_MAX_ARR] = {};
    Op::tma_arrays(p, ptr);
    for (int a = 0; a < Op::TMA_N; ++a) {
        if (!ptr[a]) continue;
        if (((uintptr_t)ptr[a] & 15) != 0 || (g.C * sizeof(typename Op::S)) % 16 != 0 ||
            !tma_encode(&td.map[a], ptr[a], sizeof(typename Op::S) == 2 ? 1 : 0, g.T, g.C, CW,
                        Ly::SR + Op::tma_extra(a)))
            return cudaErrorNotSupported;
        td.present |= 1u << a;
        td.tx_bytes += Ly::arr_bytes(a);
    }
    static int occ[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& o = occ[dev & 63];
    if (o <= 0) {
        cudaError_t e = cudaFuncSetAttribute(k_wstream<Op>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k_wstream<Op>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_wstream<Op>, 32 * Ly::NWARPS, dyn) !=
                cudaSuccess ||
            n <= 0)
            n = 1;
        o = n;
    }
    // one walker warp per walker (none when the caller asked for none), and
    // every walker's CTA resident at once: tiles are handed out only once all
    // walker roles are taken
    const uint64_t n_walk = cr.n_walk ? (uint64_t)((g.C + cr.wv - 1) / cr.wv) : 0;
    if (n_walk > (uint64_t)o * (uint64_t)sm_count()) return cudaErrorNotSupported;
    cr.n_walk = (uint32_t)n_walk;
    const uint32_t grid = persist_grid(g, cr, o);
    const uint64_t tile_bytes = (uint64_t)SB * Ly::HS;
    uint64_t d_con = ((uint64_t)LR_WS_LAG4 * grid + 3) / 4;
    const uint64_t cap = ((uint64_t)LR_STREAM_L2MB << 20) / (tile_bytes ? tile_bytes : 1);
    if (d_con > cap) d_con = cap > 1 ? cap : 1;
    g.n_draws = cr.n_walk + g.n_tiles + (uint32_t)d_con + grid - g.ticket_base;
    k_wstream<Op><<<grid, 32 * Ly::NWARPS, dyn, s>>>(p, g, cr, (uint32_t)d_con, td);
    return cudaGetLastError();
}

// Host: launch k_tchain<Op, ST> (chain protocol, TMA staging).  One tensor
// map per staged array; the ring takes ST stages of dynamic shared memory.
template <class Op, int ST>
cudaError_t launch_tchain(const typename Op::Params& p, Geom g, const Carry& cr, cudaStream_t s) {
    constexpr int L = Op::NW * Op::R, CW = 32 * Op::VEC;
    constexpr size_t dyn = (size_t)ST * tma_stage_bytes<Op>() + 128;
    static_assert(Op::TMA_N <= TMA_MAX_ARR, "too many staged arrays");
    static_assert(L + 1 <= 256 && CW <= 256, "a TMA box holds at most 256 rows and columns");
    TmaDesc td;
    memset(&td, 0, sizeof td);
    const void* ptr[TMA_MAX_ARR] = {};
    Op::tma_arrays(p, ptr);
    for (int a = 0; a < Op::TMA_N; ++a) {
        if (!ptr[a]) continue;
        if (!tma_encode(&td.map[a], ptr[a], sizeof(typename Op::S) == 2 ? 1 : 0, g.T, g.C, CW,
                        L + Op::tma_extra(a)))
            return cudaErrorInvalidValue;
        td.present |= 1u << a;
        td.tx_bytes += tma_arr_bytes<Op>(a);
    }
    static int occ[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& o = occ[dev & 63];
    if (o <= 0) {
        cudaError_t e = cudaFuncSetAttribute(k_tchain<Op, ST>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k_tchain<Op, ST>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_tchain<Op, ST>, 32 * (Op::NW + 1),
                                                          dyn) != cudaSuccess ||
            n <= 0)
            n = 1;
        o = n;
    }
    const uint32_t grid = persist_grid(g, cr, o);
    g.n_draws = g.n_tiles + grid - g.ticket_base;
    k_tchain<Op, ST><<<grid, 32 * (Op::NW + 1), dyn, s>>>(p, g, cr, td);
    return cudaGetLastError();
}

// Host: launch k_look<Op, 2> (look-back protocol, TMA staging).  Two stages:
// a tile keeps its stage until its outputs are written (the rows are read
// twice, before and after the look-back), the other one streams the CTA's
// next tile in.
template <class Op>
cudaError_t launch_look(const typename Op::Params& p, Geom g, const Carry& cr, cudaStream_t s) {
    constexpr int ST = 2;
    constexpr int L = Op::NW * Op::R, CW = 32 * Op::VEC;
    constexpr size_t dyn = (size_t)ST * tma_stage_bytes<Op>() + 128;
    static_assert(Op::TMA_N <= TMA_MAX_ARR, "too many staged arrays");
    static_assert(L + 1 <= 256 && CW <= 256, "a TMA box holds at most 256 rows and columns");
    TmaDesc td;
    memset(&td, 0, sizeof td);
    const void* ptr[TMA_MAX_ARR] = {};
    Op::tma_arrays(p, ptr);
    for (int a = 0; a < Op::TMA_N; ++a) {
        if (!ptr[a]) continue;
        if (!tma_encode(&td.map[a], ptr[a], sizeof(typename Op::S) == 2 ? 1 : 0, g.T, g.C, CW,
                        L + Op::tma_extra(a)))
            return cudaErrorInvalidValue;
        td.present |= 1u << a;
        td.tx_bytes += tma_arr_bytes<Op>(a);
    }
    static int occ[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& o = occ[dev & 63];
    if (o <= 0) {
        cudaError_t e = cudaFuncSetAttribute(k_look<Op, ST>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k_look<Op, ST>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_look<Op, ST>, 32 * Op::NW, dyn) !=
                cudaSuccess ||
            n <= 0)
            n = 1;
        o = n;
    }
    uint32_t grid = persist_grid(g, cr, o);
    // every tile fits one wave: one tile per CTA, in block order, and one
    // arrival draw each; otherwise tickets (every CTA also draws one past the end)
    const uint32_t need = g.n_tiles - g.ticket_base;
    if (need > 0 && grid >= need) {
        grid = need;
        g.n_draws = grid;
    } else {
        g.n_draws = g.n_tiles + grid - g.ticket_base;
    }
    // a programmatic dependent launch: the grid is set up while the stream's
    // previous kernel finishes (k_look waits for it before its first access)
    cudaLaunchConfig_t lc;
    memset(&lc, 0, sizeof lc);
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(32 * Op::NW);
    lc.dynamicSmemBytes = dyn;
    lc.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = LR_LOOK_PDL;
    lc.attrs = at;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, k_look<Op, ST>, p, g, cr, td);
}

// Host: launch k_cluster<Op, CL> (one cluster of n_chunks <= CL CTAs per
// channel tile), as a programmatic dependent of the stream's previous kernel.
// Up to 8 chunks the kernel is compiled for clusters of 8 (its folds and
// pushes unrolled for 8); above, for 16, which needs the non-portable opt-in.
template <class Op, int CL>
cudaError_t launch_cluster_cl(const typename Op::Params& p, const Geom& g, const Carry& cr,
                              cudaStream_t s) {
    if (CL > kClusterPortable) {
        static bool opted[64] = {false};
        int dev = 0;
        cudaGetDevice(&dev);
        if (!opted[dev & 63]) {
            const cudaError_t e =
                cudaFuncSetAttribute(k_cluster<Op, CL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
            opted[dev & 63] = true;
        }
    }
    const uint64_t grid = (uint64_t)g.n_ct * (uint64_t)g.n_chunks;
    if (grid > 0x7fffffffu) return cudaErrorInvalidValue;
    cudaLaunchConfig_t lc;
    memset(&lc, 0, sizeof lc);
    lc.gridDim = dim3((unsigned)grid);
    lc.blockDim = dim3(32 * Op::NW);
    lc.dynamicSmemBytes = 0;
    lc.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)g.n_chunks;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = LR_LOOK_PDL;
    lc.attrs = at;
    lc.numAttrs = 2;
    return cudaLaunchKernelEx(&lc, k_cluster<Op, CL>, p, g, cr);
}
template <class Op>
cudaError_t launch_cluster(const typename Op::Params& p, const Geom& g, const Carry& cr,
                           cudaStream_t s) {
    if (g.n_chunks < 1 || g.n_chunks > kClusterMax || g.n_ct < 1) return cudaErrorInvalidValue;
    if (g.n_chunks <= kClusterPortable) return launch_cluster_cl<Op, kClusterPortable>(p, g, cr, s);
    return launch_cluster_cl<Op, kClusterMax>(p, g, cr, s);
}

// Host: launch k_strip<Op, ST> when the problem has enough channel strips to
// give every resident CTA the same number of them (at most STRIP_MAX);
// returns cudaErrorNotSupported otherwise (the caller takes the chain kernel).
template <class Op, int ST, bool ONEB>
cudaError_t launch_strip(const typename Op::Params& p, const Geom& g, const Carry& cr,
                         cudaStream_t s) {
    constexpr int L = Op::NW * Op::R, CW = 32 * Op::VEC;
    constexpr size_t ring = (size_t)ST * tma_stage_bytes<Op>() + 128;
    constexpr size_t strip_bytes = 2 * 32 * Op::VEC * sizeof(float);  // two carry slots
    static int occ[64] = {0}, n_sm[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& o = occ[dev & 63];
    if (o <= 0) {
        cudaError_t e = cudaFuncSetAttribute(k_strip<Op, ST, ONEB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(ring + STRIP_MAX * strip_bytes));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k_strip<Op, ST, ONEB>,
                                 cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        int n = 0;  // residency for up to two strips per CTA
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_strip<Op, ST, ONEB>, 32 * Op::NW,
                                                          ring + 2 * strip_bytes) != cudaSuccess ||
            n <= 0)
            n = 1;
        o = n;
        cudaDeviceGetAttribute(&n_sm[dev & 63], cudaDevAttrMultiProcessorCount, dev);
    }
    const int64_t slots = (int64_t)o * (n_sm[dev & 63] > 0 ? n_sm[dev & 63] : 1);
    if (g.n_ct < kStripMinStrips || g.n_ct > slots * STRIP_MAX || g.max_grid != 0)
        return cudaErrorNotSupported;
    const int64_t m = (g.n_ct + slots - 1) / slots;
    const uint32_t G = (uint32_t)((g.n_ct + m - 1) / m);
    TmaDesc td;
    memset(&td, 0, sizeof td);
    const void* ptr[TMA_MAX_ARR] = {};
    Op::tma_arrays(p, ptr);
    for (int a = 0; a < Op::TMA_N; ++a) {
        if (!ptr[a]) continue;
        if (!tma_encode(&td.map[a], ptr[a], sizeof(typename Op::S) == 2 ? 1 : 0, g.T, g.C, CW,
                        L + Op::tma_extra(a)))
            return cudaErrorInvalidValue;
        td.present |= 1u << a;
        td.tx_bytes += tma_arr_bytes<Op>(a);
    }
    // no CTA waits for another, so the grid need not be co-resident
    k_strip<Op, ST, ONEB><<<G, 32 * Op::NW, ring + (size_t)m * strip_bytes, s>>>(p, g, cr.err, G,
                                                                                 td);
    return cudaGetLastError();
}

// Host: launch k_seg1<Op, 2> (consume only) on the segments sg.
template <class Op>
cudaError_t launch_seg1(const typename Op::Params& p, Geom g, const Carry& cr, const SegGeom& sg,
                        const TmaDesc& td, cudaStream_t s) {
    constexpr int ST = 2;
    constexpr size_t dyn = (size_t)ST * tma_stage_bytes<Op>() + 128;
    static_assert(ST <= 2, "the launch keeps SEG >= 2 >= ST");
    static int occ[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& o = occ[dev & 63];
    if (o <= 0) {
        cudaError_t e = cudaFuncSetAttribute(k_seg1<Op, ST>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k_seg1<Op, ST>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_seg1<Op, ST>, 32 * Op::NW, dyn) !=
                cudaSuccess ||
            n <= 0)
            n = 1;
        o = n;
    }
    const uint32_t grid = persist_grid(g, cr, o);
    g.n_draws = sg.n_units + grid - g.ticket_base;
    k_seg1<Op, ST><<<grid, 32 * Op::NW, dyn, s>>>(p, g, cr, sg, td);
    return cudaGetLastError();
}

// Host: launch k_seg<Op, ST> (walker protocol, segmented, TMA staging).  The
// segment length keeps the tiles between their two reads (SEG_LAG + 1
// segments per CTA) within an L2 budget.
template <class Op, int ST>
cudaError_t launch_seg(const typename Op::Params& p, Geom g, const Carry& cr, cudaStream_t s) {
    constexpr int L = Op::NW * Op::R, CW = 32 * Op::VEC;
    constexpr uint32_t SB = tma_stage_bytes<Op>();
    constexpr size_t dyn = (size_t)ST * SB + 128;
    static_assert(L + 1 <= 256 && CW <= 256, "a TMA box holds at most 256 rows and columns");
    TmaDesc td;
    memset(&td, 0, sizeof td);
    const void* ptr[TMA_MAX_ARR] = {};
    Op::tma_arrays(p, ptr);
    for (int a = 0; a < Op::TMA_N; ++a) {
        if (!ptr[a]) continue;
        if (!tma_encode(&td.map[a], ptr[a], sizeof(typename Op::S) == 2 ? 1 : 0, g.T, g.C, CW,
                        L + Op::tma_extra(a)))
            return cudaErrorInvalidValue;
        td.present |= 1u << a;
        td.tx_bytes += tma_arr_bytes<Op>(a);
    }
    static int occ[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& o = occ[dev & 63];
    if (o <= 0) {
        cudaError_t e = cudaFuncSetAttribute(k_seg<Op, ST>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k_seg<Op, ST>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_seg<Op, ST>, 32 * Op::NW, dyn) !=
                cudaSuccess ||
            n <= 0)
            n = 1;
        o = n;
    }
    const uint32_t grid = persist_grid(g, cr, o);
    const uint64_t tile_ctas = grid > cr.n_walk ? grid - cr.n_walk : 1;
    // SEG_LAG + 1 segments per CTA are in L2 at a time
    // (launches that publish the next launch's aggregates -- the DEER
    // iterations, consume-only and read once -- size their segments for the
    // walkers' and the tickets' overheads, not for L2 residency, and in rows:
    // bf16 stages count as fp32 ones)
    constexpr bool NXT = has_next_agg<Op>::value;
    const uint64_t budget = NXT ? LR_SEG1_L2MB : LR_SEG_L2MB;
    const uint64_t sb = NXT ? (uint64_t)SB * 4 / sizeof(typename Op::S) : (uint64_t)SB;
    uint64_t seg = (budget << 20) / ((SEG_LAG + 1) * tile_ctas * sb);
    if (seg < (uint64_t)ST) seg = ST;  // the ring's look-ahead stays within one iteration
    if (seg < 2) seg = 2;
    if (seg > 64) seg = 64;
    SegGeom sg;
    sg.seg = (uint32_t)seg;
    sg.n_seg = (uint32_t)((g.n_chunks + seg - 1) / seg);
    sg.n_units = sg.n_seg * (uint32_t)g.n_ct;
    // The consume-only kernel takes the segments this geometry gives (the
    // previous launch published its aggregates for them), its own grid; the
    // reduce-only pass the streaming reduction, which needs no stages.
    if constexpr (has_next_agg<Op>::value) {
        if (Op::next_agg(p).pre) return launch_seg1<Op>(p, g, cr, sg, td, s);
        if (Op::next_agg(p).reduce_only && LR_SEGRED) {
            static int occ_r[64] = {0};
            int& orr = occ_r[dev & 63];
            if (orr <= 0) {
                int n = 0;
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_segred<Op>, 32 * Op::NW, 0) !=
                        cudaSuccess ||
                    n <= 0)
                    n = 1;
                orr = n;
            }
            const uint32_t gr = (uint32_t)std::min<uint64_t>(
                (uint64_t)orr * (uint64_t)sm_count(), (uint64_t)std::max<uint32_t>(sg.n_units, 1u));
            g.n_draws = gr;  // one draw per CTA
            k_segred<Op><<<gr, 32 * Op::NW, 0, s>>>(p, g, cr, sg);
            return cudaGetLastError();
        }
    }
    // walkers draw once; a segment CTA draws until one past the end
    g.n_draws = sg.n_units + grid - g.ticket_base;
    k_seg<Op, ST><<<grid, 32 * Op::NW, dyn, s>>>(p, g, cr, sg, td);
    return cudaGetLastError();
}

// Host: launch the kernel of the launch's carry protocol; OpC / OpW / OpT / OpK
// are the operation instantiated with the tile shapes of the register chain,
// the walker, the TMA-staged kernels (strip, TMA chain) and the cluster kernel
// (void: the operation has no cluster form, and its plans never pick one).
template <class OpC, class OpW, class OpT, int ST, class OpK = void>
cudaError_t launch_persist(const typename OpC::Params& p, const Geom& g, const Carry& cr,
                           cudaStream_t s) {
    static_assert(std::is_same<typename OpC::Params, typename OpW::Params>::value &&
                      std::is_same<typename OpC::Params, typename OpT::Params>::value,
                  "all instantiations take the same arguments");
    if (cr.mode == CARRY_CLUSTER) {
        if constexpr (std::is_void<OpK>::value) return cudaErrorNotSupported;
        else return launch_cluster<OpK>(p, g, cr, s);
    }
    if (cr.mode == CARRY_LOOK) return launch_look<OpT>(p, g, cr, s);
    if (cr.mode == CARRY_CHAIN) {
        if (cr.tma) {
            cudaError_t e;
            if constexpr (strip_one_barrier<OpT>::value) e = launch_strip<OpT, 2, true>(p, g, cr, s);
            else e = launch_strip<OpT, ST, false>(p, g, cr, s);
            if (e != cudaErrorNotSupported) return e;
            return launch_tchain<OpT, ST>(p, g, cr, s);
        }
        return launch_chain<OpC>(p, g, cr, s);
    }
    if constexpr (OpT::NW * OpT::R >= OpW::NW * OpW::R)  // as seg_walk()
        if (cr.tma) return launch_seg<OpT, ST>(p, g, cr, s);
    return launch_stream<OpW>(p, g, cr, s);
}

}  // namespace lrs
