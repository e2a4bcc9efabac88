// lr_persist.cuh -- the persistent, software-pipelined kernel shared by all
// five operations.
//
// Each CTA (after the first tickets, which make walker CTAs in the walker
// protocol) loops over tiles handed out by the ticket counter.  While it
// processes tile i -- local scan, carry wait, output pass -- the loads of tile
// i+1 are already in flight into a second register set, and the ticket of
// tile i+2 is being drawn.  The wait for a tile's carry therefore no longer
// idles the memory system: HBM keeps streaming the next tile.
//
// An operation is a policy struct `Op` providing:
//   S, VEC, NW, R, REV            storage type, channels per lane, warps, rows
//                                 per thread, reverse time (backward scans)
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

template <class Op>
__device__ __forceinline__ uint32_t process_tile(const typename Op::Params& p, const Geom& g,
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
    k_persist(typename Op::Params p, Geom g, Carry cr) {
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
    if (tk < cr.n_walk) {  // walker role: computes the chunk states
        walker<typename Op::S, Op::NW>(cr, g, tk, Op::init_ptr(p));
        return;
    }
    const uint32_t limit = cr.n_walk + g.n_tiles;
    if (tk >= limit) return;
    typename Op::Acc acc;
    Op::acc_init(acc);
    typename Op::Regs r0, r1;
    uint32_t t0 = tk - cr.n_walk;
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
        const uint32_t t1 = tk - cr.n_walk;
        if (more) Op::load(p, g, tile_coord<Op>(g, t1), r1);
        tk = process_tile<Op>(p, g, cr, t0, r0, sm, xs, acc, more, &s_ticket);
        if (!more) break;
        more = tk < limit;
        t0 = tk - cr.n_walk;
        if (more) Op::load(p, g, tile_coord<Op>(g, t0), r0);
        tk = process_tile<Op>(p, g, cr, t1, r1, sm, xs, acc, more, &s_ticket);
        if (!more) break;
    }
    Op::at_exit(p, xs, acc);
}

// Walker protocol with look-ahead: ticket X first reduces tile X (loads it
// from HBM, publishes its aggregate for the walkers, keeps nothing), then
// consumes tile X - lag (loads it again -- from L2: only `lag` tiles were read
// in between -- takes the state the walkers computed, writes the outputs).
// The walkers therefore see aggregates `lag` tiles ahead of any consumer, and
// a reduce never waits, so every wait ends.  HBM traffic stays one read of
// the inputs and one write of the outputs.
template <class Op>
__global__ void __launch_bounds__(Op::NW * 32, Op::MINB)
    k_lookahead(typename Op::Params p, Geom g, Carry cr, uint32_t lag) {
    constexpr int VEC = Op::VEC;
    __shared__ CarrySmem<VEC, Op::NW> sm;
    __shared__ typename Op::Smem xs;
    __shared__ uint32_t s_ticket;
    typename Op::Acc acc;
    Op::acc_init(acc);
    const uint32_t limit = cr.n_walk + g.n_tiles + lag;
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
        if (x < g.n_tiles) {  // look-ahead: publish the aggregate of tile x
            const TileCoord tc = tile_coord<Op>(g, x);
            Op::load(p, g, tc, regs);
            float A[VEC], B[VEC];
            Op::aggregate(p, g, tc, regs, w, A, B, false);
            tile_publish_agg<VEC, Op::NW>(sm, A, B, cr, g, tc.q, tc.c, tc.cok);
        }
        if (x >= lag && x - lag < g.n_tiles) {  // consume tile x - lag
            const uint32_t y = x - lag;
            const TileCoord tc = tile_coord<Op>(g, y);
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
            tile_carry<VEC, Op::NW>(sm, A, B, init, s, cr, g, tc.q, tc.c, tc.cok, false);
            Op::finish(p, g, tc, regs, w, s, xs, acc);
        }
    }
    if (tile_role) Op::at_exit(p, xs, acc);
}

// Resident CTAs of k_persist<Op> per SM (cached per device).
template <class Op>
int persist_occupancy() {
    static int occ[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& o = occ[dev & 63];
    if (o <= 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_persist<Op>, 32 * Op::NW, 0) !=
                cudaSuccess ||
            n <= 0)
            n = 1;
        o = n;
    }
    return o;
}

template <class Op>
int lookahead_occupancy() {
    static int occ[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& o = occ[dev & 63];
    if (o <= 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_lookahead<Op>, 32 * Op::NW, 0) !=
                cudaSuccess ||
            n <= 0)
            n = 1;
        o = n;
    }
    return o;
}

// Host: launch the kernel of the carry protocol with the grid of persist_grid;
// fills n_draws.  Walker protocol: the look-ahead lag is two tiles per tile CTA,
// capped so that the lagged tiles' inputs (about 64 MB) stay within the L2.
template <class Op>
cudaError_t launch_persist(const typename Op::Params& p, Geom g, const Carry& cr, cudaStream_t s) {
    if (cr.mode == CARRY_WALK) {
        const uint32_t grid = persist_grid(g, cr, lookahead_occupancy<Op>());
        const uint64_t tile_ctas = grid > cr.n_walk ? grid - cr.n_walk : 1;
        const uint64_t tile_bytes = (uint64_t)Op::NW * Op::R * 32 * Op::VEC * sizeof(typename Op::S) *
                                    Op::IN_ARRAYS;
        uint64_t lag = 2 * tile_ctas;
        const uint64_t cap = (64ull << 20) / (tile_bytes ? tile_bytes : 1);
        if (lag > cap) lag = cap > tile_ctas ? cap : tile_ctas;
        g.n_draws = g.n_tiles + (uint32_t)lag + grid - g.ticket_base;
        k_lookahead<Op><<<grid, 32 * Op::NW, 0, s>>>(p, g, cr, (uint32_t)lag);
        return cudaGetLastError();
    }
    const uint32_t grid = persist_grid(g, cr, persist_occupancy<Op>());
    g.n_draws = g.n_tiles + grid - g.ticket_base;
    k_persist<Op><<<grid, 32 * Op::NW, 0, s>>>(p, g, cr);
    return cudaGetLastError();
}

}  // namespace lrs
