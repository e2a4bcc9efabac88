// lr_persist.cuh -- the persistent streaming kernel shared by all five
// operations (see k_stream below).
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
//   load(p, g, tc, regs)          issue the loads of one tile
//   aggregate(p, g, tc, regs, w, A, B, side)  this thread's (A, B) over its R
//                                 rows in scan order; with side = true it also
//                                 writes the outputs that need no carry
//   finish(p, g, tc, regs, w, s, sm, acc)  output pass from the entering state s
//   at_exit(p, sm, acc)           once per tile CTA after its last tile
#pragma once

#include <type_traits>

#include "lr_launch.h"

namespace lrs {

struct TileCoord {
    int64_t q;       // chunk index in scan order
    int64_t tchunk;  // chunk index in time
    int64_t c;       // first channel of this lane
    bool cok;        // the lane's channels are inside the problem
    int64_t t0;      // time of this thread's first row (scan order)
};

template <class Op>
__device__ __forceinline__ TileCoord tile_coord(const Geom& g, uint32_t tile) {
    constexpr int L = Op::NW * Op::R, CW = 32 * Op::VEC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    TileCoord tc;
    tc.q = tile / g.n_ct;
    const int64_t j = tile % g.n_ct;
    tc.c = j * CW + lane * Op::VEC;
    tc.cok = tc.c < g.C;
    tc.tchunk = Op::REV ? g.n_chunks - 1 - tc.q : tc.q;
    tc.t0 = Op::REV ? tc.tchunk * L + (L - 1) - warp * Op::R : tc.tchunk * L + warp * Op::R;
    return tc;
}

// Time of row r (scan order) of this thread.
template <class Op>
__device__ __forceinline__ int64_t row_t(const TileCoord& tc, int r) {
    return Op::REV ? tc.t0 - r : tc.t0 + r;
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
__global__ void __launch_bounds__(Op::NW * 32, Op::MINB)
    k_stream(typename Op::Params p, Geom g, Carry cr, uint32_t d_con) {
    constexpr int VEC = Op::VEC;
    __shared__ CarrySmem<VEC, Op::NW> sm;
    __shared__ typename Op::Smem xs;
    __shared__ uint32_t s_ticket;
    typename Op::Acc acc;
    Op::acc_init(acc);
    const uint32_t limit = cr.n_walk + g.n_tiles + d_con;
    bool tile_role = false;
    while (true) {
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint32_t t = atomicAdd(cr.ticket, 1u);
            if (t == g.n_draws - 1) atomicExch(cr.ticket, 0u);
            s_ticket = t + g.ticket_base;
        }
        __syncthreads();
        const uint32_t tk = s_ticket;
        if (tk < cr.n_walk) {  // walker role
            walker<typename Op::S, Op::NW>(cr, g, tk, Op::init_ptr(p));
            return;
        }
        if (tk >= limit) break;
        tile_role = true;
        const uint32_t x = tk - cr.n_walk;
        typename Op::Regs regs;
        typename Op::Work w;
        if (x < g.n_tiles) {  // reduce: publish the aggregate
            const TileCoord tc = tile_coord<Op>(g, x);
            Op::load(p, g, tc, regs);
            float A[VEC], B[VEC];
            Op::aggregate(p, g, tc, regs, w, A, B, false);
            tile_publish_agg<VEC, Op::NW>(sm, A, B, cr, g, tc.q, tc.c, tc.cok);
        }
        if (x >= d_con && x - d_con < g.n_tiles) {  // consume
            const TileCoord tc = tile_coord<Op>(g, x - d_con);
            Op::load(p, g, tc, regs);
            float A[VEC], B[VEC];
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
    }
    if (tile_role) Op::at_exit(p, xs, acc);
}

// Chain protocol (many channel tiles, few chunks): persistent CTAs walk their
// tiles in ticket order with two register sets.  While tile i is processed
// (local scan, wait for the state after the previous chunk, output pass) the
// loads of tile i+1 are in flight and the ticket of tile i+2 is being drawn.
// The chunk chain costs about one round trip per chunk level, hidden behind
// the tiles of the other channel tiles.
template <class Op>
__device__ __forceinline__ uint32_t chain_tile(const typename Op::Params& p, const Geom& g,
                                               const Carry& cr, uint32_t tile,
                                               const typename Op::Regs& regs,
                                               CarrySmem<Op::VEC, Op::NW>& sm,
                                               typename Op::Smem& xs, typename Op::Acc& acc,
                                               bool draw, uint32_t* s_ticket) {
    constexpr int VEC = Op::VEC;
    uint32_t next = 0;
    if (draw && threadIdx.x == 0) next = atomicAdd(cr.ticket, 1u);  // latency hidden by the tile
    const TileCoord tc = tile_coord<Op>(g, tile);
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
    if (draw && threadIdx.x == 0) {
        if (next == g.n_draws - 1) atomicExch(cr.ticket, 0u);
        *s_ticket = next + g.ticket_base;
    }
    __syncthreads();  // publishes the ticket; frees the carry smem for the next tile
    return draw ? *s_ticket : 0xffffffffu;
}

template <class Op>
__global__ void __launch_bounds__(Op::NW * 32, Op::MINB)
    k_chain(typename Op::Params p, Geom g, Carry cr) {
    __shared__ CarrySmem<Op::VEC, Op::NW> sm;
    __shared__ typename Op::Smem xs;
    __shared__ uint32_t s_ticket;
    if (threadIdx.x == 0) {
        const uint32_t t = atomicAdd(cr.ticket, 1u);
        if (t == g.n_draws - 1) atomicExch(cr.ticket, 0u);
        s_ticket = t + g.ticket_base;
    }
    __syncthreads();
    uint32_t tk = s_ticket;
    const uint32_t limit = g.n_tiles;
    if (tk >= limit) return;
    typename Op::Acc acc;
    Op::acc_init(acc);
    typename Op::Regs r0, r1;
    uint32_t t0 = tk;
    Op::load(p, g, tile_coord<Op>(g, t0), r0);
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t t = atomicAdd(cr.ticket, 1u);
        if (t == g.n_draws - 1) atomicExch(cr.ticket, 0u);
        s_ticket = t + g.ticket_base;
    }
    __syncthreads();
    tk = s_ticket;
    while (true) {
        // tile t0 is loaded (r0); tk is the ticket of the next tile
        bool more = tk < limit;
        const uint32_t t1 = tk;
        if (more) {
            Op::load(p, g, tile_coord<Op>(g, t1), r1);
        }
        tk = chain_tile<Op>(p, g, cr, t0, r0, sm, xs, acc, more, &s_ticket);
        if (!more) break;
        more = tk < limit;
        t0 = tk;
        if (more) {
                    Op::load(p, g, tile_coord<Op>(g, t0), r0);
        }
        tk = chain_tile<Op>(p, g, cr, t1, r1, sm, xs, acc, more, &s_ticket);
        if (!more) break;
    }
    Op::at_exit(p, xs, acc);
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
cudaError_t launch_stream(const typename Op::Params& p, Geom g, const Carry& cr, cudaStream_t s) {
    const uint32_t grid = persist_grid(g, cr, stream_occupancy<Op>());
    const uint64_t tile_ctas = grid > cr.n_walk ? grid - cr.n_walk : 1;
    const uint64_t tile_bytes =
        (uint64_t)Op::NW * Op::R * 32 * Op::VEC * sizeof(typename Op::S) * Op::IN_ARRAYS;
    uint64_t d_con = LR_STREAM_LAG * tile_ctas;
    const uint64_t cap = (32ull << 20) / (tile_bytes ? tile_bytes : 1);
    if (d_con > cap) d_con = cap > 1 ? cap : 1;
    g.n_draws = g.n_tiles + (uint32_t)d_con + grid - g.ticket_base;
    k_stream<Op><<<grid, 32 * Op::NW, 0, s>>>(p, g, cr, (uint32_t)d_con);
    return cudaGetLastError();
}

// Host: launch the kernel of the launch's carry protocol; OpC / OpW are the
// operation instantiated with the chain / walker tile shapes.
template <class OpC, class OpW>
cudaError_t launch_persist(const typename OpC::Params& p, const Geom& g, const Carry& cr,
                           cudaStream_t s) {
    static_assert(std::is_same<typename OpC::Params, typename OpW::Params>::value,
                  "both instantiations take the same arguments");
    if (cr.mode == CARRY_CHAIN) return launch_chain<OpC>(p, g, cr, s);
    return launch_stream<OpW>(p, g, cr, s);
}

}  // namespace lrs
