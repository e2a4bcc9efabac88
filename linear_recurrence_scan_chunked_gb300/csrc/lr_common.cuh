// lr_common.cuh -- device machinery shared by every chunked-scan kernel:
// storage packs (fp32 / bf16, 16-byte vectors), the tile ticket, and the
// single-pass carry of the recurrence state across time chunks.
//
// The scan is the one of page [P1] "CUDA并行化RNN训练：从O(T)到O(log T)的工程实践与
// 参数调优" (parallel-scan paragraph: an associative operation evaluated by
// divide and conquer) and page [P2] "RNN CUDA内核优化：实现序列长度无关的恒定推理延迟"
// (LSTM paragraph: tree reduction in log2 T stages; memory paragraph: shared
// memory tiling, coalesced access, no divergence at warp boundaries).  The
// operator on pairs is (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2), earlier on the
// left; a pair (A, B) is the affine map s -> A s + B.
//
// GB300 layout of the work:
//   * the sequence is [T, C] with C = B*D channels contiguous;
//   * a tile is L = NW*R time rows x CW = 32*VEC channels;  lane l of every warp
//     owns channels [l*VEC, l*VEC+VEC) of the tile (4 channels: a 16-byte fp32
//     or 8-byte bf16 vector per row, so one warp row is one contiguous 512 /
//     256-byte segment), warp w owns the R consecutive rows [w*R, w*R+R) in
//     scan order;
//   * each thread scans its R rows sequentially in registers (depth R), the NW
//     warp aggregates are combined through shared memory (depth NW), and the
//     state between time chunks comes from one of three single-pass schemes:
//       STRIP -- a CTA owns whole channel strips and walks them through time:
//                the state stays in its shared memory (wide problems);
//       CHAIN -- tile q waits for the state after chunk q-1 and publishes the
//                state after chunk q.  One L2 round trip per chunk level;
//       WALK  -- tiles (or segments of tiles) publish their aggregate (A, B)
//                and wait for the state before them, which dedicated walker
//                CTAs compute: a warp owns a few channels, its lanes own
//                WALK_P consecutive chunks each, and a Kogge-Stone prefix over
//                the lanes' folds plus the carried state gives a window of
//                32*WALK_P states at once.  For long sequences with few
//                channels (the chain would cost one round trip per chunk).
//     All fix the association of every floating-point operation by position
//     alone, so results are bitwise reproducible run to run.
//   * every published value is a self-validating 64-bit packet (value << 32 |
//     epoch): no memory fence sits on the critical path, and packets left by
//     earlier launches (older epochs) are simply not accepted;
//   * tiles (and walkers, which take the first tickets) are handed out by an
//     atomic ticket, so every producer a CTA waits for is already running: the
//     wait always ends.  Every wait is still bounded (spin_limit polls); when
//     it runs out the CTA records LR_ERR_TIMEOUT and publishes NaN, so nothing
//     downstream waits in turn;
//   * the launch's epoch lives on the device, in the high half of the 64-bit
//     ticket word (the low half counts the tickets): every draw returns both,
//     so a CTA learns its launch's epoch with its first ticket at no extra
//     cost, and the last drawer retires the epoch as it resets the counter.
//     A launch replayed from a CUDA graph therefore takes a fresh epoch, like
//     one enqueued by the host.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace lrs {

constexpr uint32_t ERRBIT_TIMEOUT = 1u;
constexpr int CARRY_CHAIN = 0;
constexpr int CARRY_WALK = 1;
constexpr int CARRY_LOOK = 2;
constexpr int CARRY_CLUSTER = 3;  // one thread-block cluster per channel tile (short problems)
constexpr int WALK_MAX_WV = 4;  // channels per walker warp (upper bound)
constexpr int WALK_P = 4;       // consecutive chunks per walker lane

typedef unsigned long long u64;

// Carry-protocol state of one launch.
// Unroll factor of the warp-aggregate folds (a warp folds the aggregates of
// the warps before it: a dependent chain whose shared-memory loads an unrolled
// loop issues ahead).
#ifndef LR_FOLD_UNROLL
#define LR_FOLD_UNROLL 1
#endif
constexpr int kFoldUnroll = LR_FOLD_UNROLL;

struct Carry {
    u64* agg;             // WALK: [C][n_chunks][2] packets (A, B) of every tile;
                          // LOOK: [n_chunks][C][2] (chunk-major: a tile publishes
                          // one contiguous row, a look-back reads whole rows)
    u64* inc;             // packets: state after chunk q (scan order); CHAIN stores
                          // them chunk-major [n_chunks][C] (a tile reads one row),
                          // WALK channel-major [C][n_chunks] (a walker warp reads
                          // and writes 32 consecutive chunks of one channel)
    u64* tk;              // ticket word: low 32 bits the ticket counter (0 between
                          // launches), high 32 bits the last retired epoch
    uint32_t* err;        // sticky error bits
    uint32_t epoch;       // this launch's epoch (1 .. 2^32-1): set on the device
                          // from the ticket word by each CTA's first draw
    uint32_t spin_limit;  // polls before a wait gives up
    int mode;             // CARRY_CHAIN, CARRY_WALK, CARRY_LOOK or CARRY_CLUSTER
    uint32_t n_walk;      // walker CTAs (first tickets); 0 in CHAIN / LOOK mode
    int wv;               // channels per walker warp (WALK)
    int tma;              // CHAIN: tiles are staged by TMA (k_strip / k_tchain)
};

// Aggregates published one launch ahead, for operations whose next launch
// builds its coefficients from this launch's outputs (segmented walker
// kernel only).
struct NextAgg {
    u64* agg;              // [C][n_seg][2] (A, B) packets of the next launch; nullptr: none
    uint32_t epoch;        // the next launch's epoch (set on the device)
    uint32_t pre;          // this launch's aggregates were published by the previous launch
    uint32_t reduce_only;  // this launch only publishes the next launch's aggregates (from its
                           // own coefficients: the pass before a solve's first iteration)
};
// Op::NEXT_AGG (optional, default false): the operation computes the next
// launch's per-thread aggregate in finish() (Work::NA, Work::NB) and exposes
// its NextAgg through Op::next_agg(params).
template <class Op, class = void>
struct has_next_agg : std::false_type {};
template <class Op>
struct has_next_agg<Op, std::void_t<decltype(Op::NEXT_AGG)>>
    : std::integral_constant<bool, Op::NEXT_AGG> {};

// Op::STRIP_ONE_BARRIER (optional, default false): the strip kernel runs the
// operation with one barrier per tile (two stages, double-buffered warp
// aggregates) -- for operations whose per-tile work, not HBM, bounds a CTA.
template <class Op, class = void>
struct strip_one_barrier : std::false_type {};
template <class Op>
struct strip_one_barrier<Op, std::void_t<decltype(Op::STRIP_ONE_BARRIER)>>
    : std::integral_constant<bool, Op::STRIP_ONE_BARRIER> {};

// Op::STREAM_WS: the walker protocol's streaming launches take the
// warp-specialised TMA kernel (k_wstream) where it applies.
template <class Op, class = void>
struct stream_ws : std::false_type {};
template <class Op>
struct stream_ws<Op, std::void_t<decltype(Op::STREAM_WS)>>
    : std::integral_constant<bool, Op::STREAM_WS> {};

struct Geom {
    int64_t T;            // rows
    int64_t C;            // channels (B*D)
    int64_t D;            // features (per-feature parameters use c % D)
    int64_t n_chunks;     // ceil(T / L)
    int n_ct;             // ceil(C / CW)
    uint32_t n_tiles;     // n_chunks * n_ct
    uint32_t n_draws;     // tickets drawn by the whole launch (the last drawer resets)
    uint32_t ticket_base; // added to every ticket (the timeout test starts past tile 0)
    uint32_t max_grid;    // 0, or an upper bound on the CTAs launched (timeout test)
    // c / D without a 64-bit division (per-feature parameters, per-sequence
    // state): while C < 2^31, c / D = (umulhi(c, d_mul) + c) >> d_shift, the
    // round-up multiplier of Granlund and Montgomery ("Division by invariant
    // integers using multiplication", 1994); d_mul = 0: plain division.
    uint32_t d_mul;
    uint32_t d_shift;
};

// Host: the multiplier and shift of c / D (0 when C or D is out of range).
inline void set_channel_div(Geom& g) {
    g.d_mul = 0;
    g.d_shift = 0;
    if (g.D < 1 || g.D >= ((int64_t)1 << 31) || g.C >= ((int64_t)1 << 31)) return;
    uint32_t s = 0;
    while (((uint64_t)1 << s) < (uint64_t)g.D) ++s;
    // floor(2^32 (2^s - D) / D) + 1 < 2^32, since 2^s - D < D
    g.d_mul = (uint32_t)((((uint64_t)1 << 32) * (((uint64_t)1 << s) - (uint64_t)g.D)) / (uint64_t)g.D + 1);
    g.d_shift = s;
}

// Channel c's feature index c mod D and sequence index c / D.
__host__ __device__ __forceinline__ int64_t chan_seq(const Geom& g, int64_t c) {
    if (g.d_mul == 0) return c / g.D;
#ifdef __CUDA_ARCH__
    const uint32_t hi = __umulhi((uint32_t)c, g.d_mul);
#else
    const uint32_t hi = (uint32_t)(((uint64_t)(uint32_t)c * g.d_mul) >> 32);
#endif
    return (int64_t)(((uint64_t)hi + (uint32_t)c) >> g.d_shift);
}
__host__ __device__ __forceinline__ int64_t chan_feat(const Geom& g, int64_t c) {
    return c - chan_seq(g, c) * g.D;
}

// Barrier of the NW consumer warps of a CTA (named barrier 1).  The scan
// kernels that stage tiles with TMA add a producer warp that never takes part
// in the tile arithmetic; in the other kernels NW*32 is the whole CTA.
template <int NW>
__device__ __forceinline__ void csync() {
    asm volatile("bar.sync 1, %0;" ::"r"(NW * 32) : "memory");
}

// Programmatic dependent launch (sm_90+): wait until the grids this one
// depends on have completed and their memory operations are visible; let the
// grids that depend on this one be scheduled.  Both are no-ops for a grid
// launched without the programmatic attribute.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------- memory ops

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// ------------------------------------------------------ tickets and epochs
// The epoch that follows the last retired one (0 is never an epoch: a packet
// buffer cleared to zero holds no valid packet).
__host__ __device__ __forceinline__ uint32_t epoch_after(uint32_t last) {
    return last + 1u == 0u ? 1u : last + 1u;
}
// Draw one ticket: returns it, and sets c.epoch to the launch's epoch (every
// draw of a launch sees the same high half, until the last drawer retires it).
template <class Cr>
__device__ __forceinline__ uint32_t draw_ticket(Cr& c) {
    const unsigned long long v =
        atomicAdd(reinterpret_cast<unsigned long long*>(c.tk), 1ull);
    c.epoch = epoch_after((uint32_t)(v >> 32));
    return (uint32_t)v;
}
// After ticket t was drawn: the launch's last draw resets the counter and
// retires the epoch in one atomic (every CTA has drawn by then, so each has
// read the epoch).  A maximum rather than an exchange: when a wait of this
// launch ran out and already retired later epochs, the word keeps them (and
// its counter, which lr_last_error resets) -- except at the wrap to epoch 1.
template <class Cr, class G>
__device__ __forceinline__ void ticket_drawn(const Cr& c, const G& g, uint32_t t) {
    if (t == g.n_draws - 1) {
        unsigned long long* w = reinterpret_cast<unsigned long long*>(c.tk);
        const unsigned long long v = (unsigned long long)c.epoch << 32;
        if (c.epoch == 1u) atomicExch(w, v);
        else atomicMax(w, v);
    }
}
// Retire the launch's epoch outside the normal end of a launch: a wait that
// ran out (the launch will not complete its draws) or a launch with nothing
// to do.  The counter half is left alone; a timed-out launch leaves it for
// lr_last_error to reset.  Several callers in one launch only skip epochs.
template <class Cr>
__device__ __forceinline__ void retire_epoch(const Cr& c) {
    atomicAdd(reinterpret_cast<unsigned long long*>(c.tk), 1ull << 32);
}
// A wait ran out: record the error, retire the epoch.
template <class Cr>
__device__ __forceinline__ void give_up(const Cr& c) {
    atomicOr(c.err, ERRBIT_TIMEOUT);
    retire_epoch(c);
}

// Streaming 16-byte loads of read-once inputs (no L1 allocation).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ uint2 ld_stream_u2(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}
// L2 eviction-priority policies (createpolicy) and loads that carry one: the
// walker-protocol kernel reads every tile twice, and the second read should
// find it in L2.
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ld_hint_u4(const void* p, uint64_t pol) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ uint2 ld_hint_u2(const void* p, uint64_t pol) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ uint32_t ld_hint_b32(const void* p, uint64_t pol) {
    uint32_t r;
    asm volatile("ld.global.nc.L2::cache_hint.b32 %0, [%1], %2;" : "=r"(r) : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ uint32_t ld_hint_u16(const void* p, uint64_t pol) {
    unsigned short r;
    asm volatile("ld.global.nc.L2::cache_hint.u16 %0, [%1], %2;" : "=h"(r) : "l"(p), "l"(pol));
    return (uint32_t)r;
}
// Output stores are streaming (.cs: evict-first in L2): outputs are not
// read back by the launch that writes them, and tiles parked in L2 for a
// second read (walker-protocol kernels) or the next iterate's inputs keep
// their lines.  0: plain stores.
#ifndef LR_ST_CS
#define LR_ST_CS 1
#endif
__device__ __forceinline__ void st_u2(void* p, uint2 v) {
#if LR_ST_CS
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
#else
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
#endif
}
__device__ __forceinline__ void st_u4(void* p, uint4 v) {
#if LR_ST_CS
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
#else
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
#endif
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t bf_bits(float x) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ uint32_t bf_pack(float lo, float hi) {
    return bf_bits(lo) | (bf_bits(hi) << 16);
}

// --------------------------------------------------------- storage packs
// Pack<S, VEC>: VEC consecutive elements of storage type S held in registers
// (bf16 kept packed, two per 32-bit register).  VEC * sizeof(S) is 16 bytes on
// the vector path and one element on the scalar path (the cluster kernel also
// takes two-element packs on the vector path).

template <typename S, int VEC>
struct Pack;

template <int VEC>
struct Pack<float, VEC> {
    static_assert(VEC == 4 || VEC == 2 || VEC == 1, "fp32 packs hold 4, 2 or 1 elements");
    float v[VEC];
    __device__ __forceinline__ void load(const float* p) {
        if constexpr (VEC == 4) {
            uint4 r = ld_stream_u4(p);
            v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
            v[2] = __uint_as_float(r.z); v[3] = __uint_as_float(r.w);
        } else if constexpr (VEC == 2) {
            const uint2 r = ld_stream_u2(p);
            v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
        } else {
            v[0] = __ldg(p);
        }
    }
    __device__ __forceinline__ void load_hint(const float* p, uint64_t pol) {
        if constexpr (VEC == 4) {
            uint4 r = ld_hint_u4(p, pol);
            v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
            v[2] = __uint_as_float(r.z); v[3] = __uint_as_float(r.w);
        } else if constexpr (VEC == 2) {
            const uint2 r = ld_hint_u2(p, pol);
            v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
        } else {
            v[0] = __uint_as_float(ld_hint_b32(p, pol));
        }
    }
    __device__ __forceinline__ void load_shared(const float* p) {
        if constexpr (VEC == 4) {
            const float4 f = *reinterpret_cast<const float4*>(p);
            v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
        } else if constexpr (VEC == 2) {
            const float2 f = *reinterpret_cast<const float2*>(p);
            v[0] = f.x; v[1] = f.y;
        } else {
            v[0] = *p;
        }
    }
    __device__ __forceinline__ float get(int i) const { return v[i]; }
    __device__ __forceinline__ void ident(float x) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) v[i] = x;
    }
};

template <int VEC>
struct Pack<__nv_bfloat16, VEC> {
    static_assert(VEC == 8 || VEC == 4 || VEC == 2 || VEC == 1, "bf16 packs hold 8, 4, 2 or 1 elements");
    static constexpr int NW_ = VEC == 1 ? 1 : VEC / 2;
    uint32_t w[NW_];
    __device__ __forceinline__ void load(const __nv_bfloat16* p) {
        if constexpr (VEC == 8) {
            uint4 r = ld_stream_u4(p);
            w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
        } else if constexpr (VEC == 4) {
            const uint2 r = ld_stream_u2(p);
            w[0] = r.x; w[1] = r.y;
        } else if constexpr (VEC == 2) {
            w[0] = __ldg(reinterpret_cast<const unsigned int*>(p));
        } else {
            w[0] = (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p));
        }
    }
    __device__ __forceinline__ void load_hint(const __nv_bfloat16* p, uint64_t pol) {
        if constexpr (VEC == 8) {
            uint4 r = ld_hint_u4(p, pol);
            w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
        } else if constexpr (VEC == 4) {
            const uint2 r = ld_hint_u2(p, pol);
            w[0] = r.x; w[1] = r.y;
        } else if constexpr (VEC == 2) {
            w[0] = ld_hint_b32(p, pol);
        } else {
            w[0] = ld_hint_u16(p, pol);
        }
    }
    __device__ __forceinline__ void load_shared(const __nv_bfloat16* p) {
        if constexpr (VEC == 8) {
            const uint4 r = *reinterpret_cast<const uint4*>(p);
            w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
        } else if constexpr (VEC == 4) {
            const uint2 r = *reinterpret_cast<const uint2*>(p);
            w[0] = r.x; w[1] = r.y;
        } else if constexpr (VEC == 2) {
            w[0] = *reinterpret_cast<const uint32_t*>(p);
        } else {
            w[0] = (uint32_t)*reinterpret_cast<const unsigned short*>(p);
        }
    }
    __device__ __forceinline__ float get(int i) const {
        if constexpr (VEC > 1) return (i & 1) ? bf_hi(w[i >> 1]) : bf_lo(w[i >> 1]);
        else return bf_lo(w[0]);
    }
    __device__ __forceinline__ void ident(float x) {
        uint32_t b = bf_bits(x);
#pragma unroll
        for (int i = 0; i < NW_; ++i) w[i] = VEC > 1 ? (b | (b << 16)) : b;
    }
};

// Store VEC fp32 values to storage type S (bf16: round to nearest-even).
template <typename S, int VEC>
__device__ __forceinline__ void store_vec(S* p, const float (&x)[VEC]) {
    if constexpr (sizeof(S) == 4) {
        if constexpr (VEC == 4)
            st_u4(p, make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]),
                                __float_as_uint(x[2]), __float_as_uint(x[3])));
        else if constexpr (VEC == 2)
            st_u2(p, make_uint2(__float_as_uint(x[0]), __float_as_uint(x[1])));
        else
            *reinterpret_cast<float*>(p) = x[0];
    } else {
        if constexpr (VEC == 8)
            st_u4(p, make_uint4(bf_pack(x[0], x[1]), bf_pack(x[2], x[3]), bf_pack(x[4], x[5]),
                                bf_pack(x[6], x[7])));
        else if constexpr (VEC == 4)
            st_u2(p, make_uint2(bf_pack(x[0], x[1]), bf_pack(x[2], x[3])));
        else if constexpr (VEC == 2)
            *reinterpret_cast<uint32_t*>(p) = bf_pack(x[0], x[1]);
        else
            *reinterpret_cast<unsigned short*>(p) = (unsigned short)bf_bits(x[0]);
    }
}

// Load VEC values of storage type S into fp32 (for small per-state tensors).
template <typename S, int VEC>
__device__ __forceinline__ void load_vec(const S* p, float (&x)[VEC]) {
    Pack<S, VEC> pk;
    pk.load(p);
#pragma unroll
    for (int i = 0; i < VEC; ++i) x[i] = pk.get(i);
}

// fp32 parameter vector (w, bf, br): VEC consecutive floats, 16-byte aligned
// on the vector path.
template <int VEC>
__device__ __forceinline__ void load_param(const float* p, float (&x)[VEC]) {
    if constexpr (VEC >= 4) {
#pragma unroll
        for (int i = 0; i < VEC; i += 4) {
            float4 f = __ldg(reinterpret_cast<const float4*>(p + i));
            x[i] = f.x; x[i + 1] = f.y; x[i + 2] = f.z; x[i + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) x[i] = __ldg(p + i);
    }
}

// ------------------------------------------------------------------ packets

__device__ __forceinline__ u64 pkt(float v, uint32_t e) {
    return ((u64)__float_as_uint(v) << 32) | e;
}
__device__ __forceinline__ float pkt_val(u64 p) { return __uint_as_float((uint32_t)(p >> 32)); }
__device__ __forceinline__ bool pkt_ok(u64 p, uint32_t e) { return (uint32_t)p == e; }

__device__ __forceinline__ void ld_pkt2(const u64* p, u64& a, u64& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ u64 ld_pkt(const u64* p) {
    u64 a;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(a) : "l"(p) : "memory");
    return a;
}
__device__ __forceinline__ void st_pkt2(u64* p, u64 a, u64 b) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1,%2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void st_pkt(u64* p, u64 a) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(a) : "memory");
}

// L2-only (.cg) packet accesses for the walker's hot loop: coalesced across
// the warp, never served from a stale L1 line; an aligned 8-byte access is
// never torn, and a packet is only accepted when its epoch matches.
__device__ __forceinline__ void ld_pkt2_cg(const u64* p, u64& a, u64& b) {
    asm volatile("ld.global.cg.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ u64 ld_pkt_cg(const u64* p) {
    u64 a;
    asm volatile("ld.global.cg.u64 %0, [%1];" : "=l"(a) : "l"(p) : "memory");
    return a;
}
__device__ __forceinline__ void st_pkt_cg(u64* p, u64 a) {
    asm volatile("st.global.cg.u64 [%0], %1;" ::"l"(p), "l"(a) : "memory");
}

// VEC state packets of one lane (16-byte aligned when VEC is even).
template <int VEC>
__device__ __forceinline__ void put_states(u64* p, const float (&x)[VEC], uint32_t e) {
    if constexpr (VEC % 2 == 0) {
#pragma unroll
        for (int i = 0; i < VEC; i += 2) st_pkt2(p + i, pkt(x[i], e), pkt(x[i + 1], e));
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) st_pkt(p + i, pkt(x[i], e));
    }
}
template <int VEC>
__device__ __forceinline__ bool get_states(const u64* p, float (&x)[VEC], uint32_t e) {
    bool ok = true;
    if constexpr (VEC % 2 == 0) {
#pragma unroll
        for (int i = 0; i < VEC; i += 2) {
            u64 a, b;
            ld_pkt2(p + i, a, b);
            ok = ok && pkt_ok(a, e) && pkt_ok(b, e);
            x[i] = pkt_val(a);
            x[i + 1] = pkt_val(b);
        }
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const u64 a = ld_pkt(p + i);
            ok = ok && pkt_ok(a, e);
            x[i] = pkt_val(a);
        }
    }
    return ok;
}

// VEC state packets of one lane stored `stride` packets apart (channel-major).
template <int VEC>
__device__ __forceinline__ bool get_states_strided(const u64* p, int64_t stride, float (&x)[VEC],
                                                   uint32_t e) {
    bool ok = true;
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const u64 a = ld_pkt(p + i * stride);
        ok = ok && pkt_ok(a, e);
        x[i] = pkt_val(a);
    }
    return ok;
}

// Bounded wait helper: returns true when the caller should give up.  Sleeps
// grow to max_sleep_ns between polls (0: pure spin -- a walker with an SM of its
// own, which is on every tile's critical path, must notice new aggregates at
// once).
__device__ __forceinline__ bool wait_step(const Carry& cr, uint32_t& spins, uint32_t& sleep_ns,
                                          uint32_t max_sleep_ns) {
    ++spins;
    if (spins > cr.spin_limit) return true;
    if ((spins & 63u) == 0) {
        uint32_t e;
        asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(e) : "l"(cr.err) : "memory");
        if (e & ERRBIT_TIMEOUT) return true;
    }
    if (sleep_ns) __nanosleep(sleep_ns);
    sleep_ns = sleep_ns == 0 ? (max_sleep_ns ? 16 : 0)
                             : (sleep_ns * 2 < max_sleep_ns ? sleep_ns * 2 : max_sleep_ns);
    return false;
}
constexpr uint32_t kTileMaxSleepNs = 64;

// ------------------------------------------------------------- the walker

// One walker CTA (NW warps).  Warp gw = wid*NW + warp owns channels
// [gw*wv, gw*wv + wv).  It sweeps the chunks in windows of 32*WALK_P: lane l
// owns the WALK_P consecutive chunks w0 + l*WALK_P + k.  With every
// aggregate of a window loaded in one round trip, it forms each lane's left
// fold over its chunks, an inclusive Kogge-Stone prefix of those folds across
// the lanes, and then, lane by lane, the chunk states
//     state(q) = a_q * state(q-1) + b_q   from the lane's entering state
// s_l = E_l.A * s_in + E_l.B (E_l: exclusive prefix, s_in: state after the
// previous window).  The association of every operation depends on the chunk
// index only, so the states are bitwise reproducible.  States are published
// as soon as the aggregates before them are visible -- a lane whose later
// chunks are not visible yet still publishes its leading ones -- so no tile
// ever waits for a tile with a larger ticket.  A warp of one channel (MV = 1)
// loads the next window's aggregates while it folds the current one, so its
// windows cost compute, not a round trip each.

// Issue the loads of one window's aggregate packets (not-yet-published ones
// come back with an old epoch and are polled again).
template <int MV>
__device__ __forceinline__ void walk_load(const Carry& cr, const Geom& g, int64_t c0,
                                          const bool (&chan)[MV], int64_t q0, int n_lane,
                                          u64 (&pk)[WALK_P][MV][2]) {
#pragma unroll
    for (int k = 0; k < WALK_P; ++k)
#pragma unroll
        for (int v = 0; v < MV; ++v) {
            pk[k][v][0] = pk[k][v][1] = 0;
            if (chan[v] && k < n_lane)
                ld_pkt2_cg(cr.agg + 2 * ((c0 + v) * g.n_chunks + q0 + k), pk[k][v][0], pk[k][v][1]);
        }
}

// Fold and publish one window [w0, w0 + n_win); s_in: state before it, on
// return the state after it.
template <int MV>
__device__ __forceinline__ void walk_window(const Carry& cr, const Geom& g, int64_t c0,
                                            const bool (&chan)[MV], int wv, int64_t w0, int n_win,
                                            u64 (&pk)[WALK_P][MV][2], float (&s_in)[MV],
                                            bool& dead, uint32_t max_sleep) {
    constexpr int P = WALK_P;
    const int lane = threadIdx.x & 31;
    const int64_t q0 = w0 + (int64_t)lane * P;  // this lane's first chunk
    uint32_t spins = 0, sleep_ns = 0;
    bool okk[P];
#pragma unroll
    for (int k = 0; k < P; ++k) okk[k] = false;
    int pub = 0;  // chunks of this window already published (a prefix)
    while (true) {
        // vp: leading chunks of this lane whose aggregates are visible (chunks
        // past the end of the problem count as visible)
        int vp = 0;
        bool run = true;
#pragma unroll
        for (int k = 0; k < P; ++k) {
            bool ok = okk[k] || lane * P + k >= n_win;
            if (!ok) {
                ok = true;
#pragma unroll
                for (int v = 0; v < MV; ++v)
                    if (chan[v]) ok = ok && pkt_ok(pk[k][v][0], cr.epoch) && pkt_ok(pk[k][v][1], cr.epoch);
                okk[k] = ok;
            }
            run = run && ok;
            vp += run ? 1 : 0;
        }
        const unsigned notfull = ~__ballot_sync(0xffffffffu, vp == P);
        const int npre = notfull ? __ffs(notfull) - 1 : 32;  // leading complete lanes
        const int vp_part = __shfl_sync(0xffffffffu, vp, npre < 32 ? npre : 31);
        int limit = npre * P + (npre < 32 ? vp_part : 0);
        if (limit > n_win) limit = n_win;
        if (dead) limit = n_win;
        float s_end[MV];
        if (limit > pub) {
            float A[MV], B[MV];
#pragma unroll
            for (int v = 0; v < MV; ++v) { A[v] = 1.f; B[v] = 0.f; }
            if (lane < npre) {  // left fold over this lane's chunks
#pragma unroll
                for (int k = 0; k < P; ++k)
#pragma unroll
                    for (int v = 0; v < MV; ++v)
                        if (chan[v] && lane * P + k < n_win) {
                            const float a = pkt_val(pk[k][v][0]);
                            B[v] = __fmaf_rn(a, B[v], pkt_val(pk[k][v][1]));
                            A[v] *= a;
                        }
            }
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
                for (int v = 0; v < MV; ++v) {
                    if (v >= wv) continue;
                    const float pa = __shfl_up_sync(0xffffffffu, A[v], off);
                    const float pb = __shfl_up_sync(0xffffffffu, B[v], off);
                    if (lane >= off) {
                        B[v] = __fmaf_rn(A[v], pb, B[v]);
                        A[v] = pa * A[v];
                    }
                }
            }
            float st[MV];
#pragma unroll
            for (int v = 0; v < MV; ++v) {  // exclusive prefix -> entering state
                const float ea = __shfl_up_sync(0xffffffffu, A[v], 1);
                const float eb = __shfl_up_sync(0xffffffffu, B[v], 1);
                st[v] = lane == 0 ? s_in[v] : __fmaf_rn(ea, s_in[v], eb);
            }
#pragma unroll
            for (int k = 0; k < P; ++k) {
                const int rel = lane * P + k;
#pragma unroll
                for (int v = 0; v < MV; ++v) {
                    if (!chan[v]) continue;
                    if (rel < limit)
                        st[v] = dead ? __int_as_float(0x7fc00000)
                                     : __fmaf_rn(pkt_val(pk[k][v][0]), st[v], pkt_val(pk[k][v][1]));
                    if (rel >= pub && rel < limit)
                        st_pkt_cg(cr.inc + (c0 + v) * g.n_chunks + q0 + k, pkt(st[v], cr.epoch));
                }
            }
#pragma unroll
            for (int v = 0; v < MV; ++v) s_end[v] = st[v];
            pub = limit;
        }
        if (pub == n_win) {  // state after the window's last chunk -> next window
            const int owner = (n_win - 1) / P;
#pragma unroll
            for (int v = 0; v < MV; ++v) s_in[v] = __shfl_sync(0xffffffffu, s_end[v], owner);
            return;
        }
        if (__any_sync(0xffffffffu, wait_step(cr, spins, sleep_ns, max_sleep))) {
            if (lane == 0) give_up(cr);
            dead = true;  // publish NaN for the rest so no tile keeps waiting
            continue;
        }
#pragma unroll
        for (int k = 0; k < P; ++k)  // re-poll what was not visible
#pragma unroll
            for (int v = 0; v < MV; ++v)
                if (chan[v] && !okk[k] && lane * P + k < n_win)
                    ld_pkt2_cg(cr.agg + 2 * ((c0 + v) * g.n_chunks + q0 + k), pk[k][v][0], pk[k][v][1]);
    }
}

// Walker warp gw: channels [gw*wv, gw*wv + wv).
template <typename S, int MV>
__device__ void walker_mv(const Carry& cr, const Geom& g, int64_t gw, const S* __restrict__ init,
                          uint32_t max_sleep) {
    constexpr int P = WALK_P, WIN = 32 * WALK_P;
    const int lane = threadIdx.x & 31;
    const int64_t c0 = gw * cr.wv;
    const int64_t last = g.n_chunks - 1;  // states are needed for chunks 0 .. last-1
    if (c0 >= g.C || last <= 0) return;
    const int wv = cr.wv;
    bool chan[MV];
#pragma unroll
    for (int v = 0; v < MV; ++v) chan[v] = v < wv && c0 + v < g.C;
    float s_in[MV];
#pragma unroll
    for (int v = 0; v < MV; ++v) {
        s_in[v] = 0.f;
        if (chan[v] && init != nullptr) {
            Pack<S, 1> pk;
            pk.load(init + c0 + v);
            s_in[v] = pk.get(0);
        }
    }
    bool dead = false;  // a wait ran out: every remaining state is published as NaN
    auto n_of = [&](int64_t w0) { return (int)((last - w0) < WIN ? (last - w0) : WIN); };
    auto lane_n = [&](int n_win) {
        const int r = n_win - lane * P;
        return r < 0 ? 0 : (r > P ? P : r);
    };
    if constexpr (MV == 1) {
        // two windows in flight: the next one's loads overlap this one's fold
        u64 pa[P][MV][2], pb[P][MV][2];
        walk_load<MV>(cr, g, c0, chan, (int64_t)lane * P, lane_n(n_of(0)), pa);
        for (int64_t w0 = 0; w0 < last; w0 += 2 * WIN) {
            const int64_t w1 = w0 + WIN;
            if (w1 < last) walk_load<MV>(cr, g, c0, chan, w1 + (int64_t)lane * P, lane_n(n_of(w1)), pb);
            walk_window<MV>(cr, g, c0, chan, wv, w0, n_of(w0), pa, s_in, dead, max_sleep);
            if (w1 >= last) break;
            const int64_t w2 = w1 + WIN;
            if (w2 < last) walk_load<MV>(cr, g, c0, chan, w2 + (int64_t)lane * P, lane_n(n_of(w2)), pa);
            walk_window<MV>(cr, g, c0, chan, wv, w1, n_of(w1), pb, s_in, dead, max_sleep);
        }
    } else {
        u64 pk[P][MV][2];
        for (int64_t w0 = 0; w0 < last; w0 += WIN) {
            walk_load<MV>(cr, g, c0, chan, w0 + (int64_t)lane * P, lane_n(n_of(w0)), pk);
            walk_window<MV>(cr, g, c0, chan, wv, w0, n_of(w0), pk, s_in, dead, max_sleep);
        }
    }
}

template <typename S>
__device__ void walker_warp(const Carry& cr, const Geom& g, int64_t gw, const S* __restrict__ init,
                            uint32_t max_sleep = 0) {
    if (cr.wv == 1) walker_mv<S, 1>(cr, g, gw, init, max_sleep);
    else walker_mv<S, WALK_MAX_WV>(cr, g, gw, init, max_sleep);
}
// Warp w of walker CTA wid is walker warp wid*NW + w.
template <typename S, int NW>
__device__ void walker(const Carry& cr, const Geom& g, uint32_t wid, const S* __restrict__ init) {
    walker_warp<S>(cr, g, (int64_t)wid * NW + (threadIdx.x >> 5), init);
}

// -------------------------------------------------------------- the tile

// Shared memory for combining the NW warp aggregates of a tile.
template <int VEC, int NW>
struct CarrySmem {
    float a[NW][32][VEC];
    float b[NW][32][VEC];
    float carry[32][VEC];
};

// Whole CTA.  (A, B): this thread's aggregate over its R rows (scan order).
// init: state before the whole scan (used by warp 0 when q == 0).  c: first
// channel of this lane, cok: it is inside the problem.  Returns in `start` the
// state entering this thread's first row.  Chain protocol: publishes the
// state after this chunk, INC(q).  Walker protocol: the tile's aggregate was
// published by tile_publish_agg; the entering state comes from the walkers.
template <int VEC, int NW>
__device__ __forceinline__ void tile_carry(CarrySmem<VEC, NW>& sm, const float (&A)[VEC],
                                           const float (&B)[VEC], const float (&init)[VEC],
                                           float (&start)[VEC], const Carry& cr, const Geom& g,
                                           int64_t q, int64_t c, bool cok,
                                           const u64* pre = nullptr) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        sm.a[warp][lane][v] = A[v];
        sm.b[warp][lane][v] = B[v];
    }
    csync<NW>();
    if (warp == 0) {
        float TA[VEC], TB[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { TA[v] = 1.f; TB[v] = 0.f; }
#pragma unroll
        for (int w = 0; w < NW; ++w)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float a = sm.a[w][lane][v], b = sm.b[w][lane][v];
                TB[v] = __fmaf_rn(a, TB[v], b);
                TA[v] *= a;
            }
        constexpr int CW = 32 * VEC;
        float cin[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) cin[v] = 0.f;
        const bool more = q < g.n_chunks - 1;  // a later chunk needs this one's state
        const int64_t base = q * g.C + c;
        const bool walk = cr.mode == CARRY_WALK;
        if (q == 0) {
            if (cok) {
#pragma unroll
                for (int v = 0; v < VEC; ++v) cin[v] = init[v];
            }
        } else {
            // Packets loaded early by the caller (warp 0, this lane's channels of
            // chunk q-1): when they all carry this launch's epoch, no poll at all.
            bool have = false;
            if (pre != nullptr) {
                bool ok = true;
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    ok = ok && (!cok || pkt_ok(pre[v], cr.epoch));
                    cin[v] = pkt_val(pre[v]);
                }
                have = __all_sync(0xffffffffu, ok);
            }
            // Lane 0 polls one packet, the state of one channel of the tile; once it
            // is there every lane reads its own.  One 8-byte poll per tile keeps the
            // L2 free for the data, and the polled channel rotates with the chunk
            // so that neighbouring tiles never poll the same cache line.
            const int64_t c_first = c - lane * VEC;
            int64_t n_tile_ch = g.C - c_first;
            if (n_tile_ch > CW) n_tile_ch = CW;
            const int64_t c_rep = c_first + (int64_t)((q * 37) % n_tile_ch);
            const u64* rep = walk ? cr.inc + c_rep * g.n_chunks + q - 1 : cr.inc + (q - 1) * g.C + c_rep;
            uint32_t spins = 0, sleep_ns = 0;
            while (!have) {
                // chain: the states are one contiguous row, read directly (one
                // round trip when they are there already, the common case)
                bool rep_ok = !walk;
                if (walk && lane == 0) rep_ok = pkt_ok(ld_pkt(rep), cr.epoch);
                if (__shfl_sync(0xffffffffu, rep_ok, 0)) {
                    const bool ok =
                        !cok || (walk ? get_states_strided<VEC>(cr.inc + c * g.n_chunks + q - 1,
                                                                 g.n_chunks, cin, cr.epoch)
                                      : get_states<VEC>(cr.inc + base - g.C, cin, cr.epoch));
                    if (__all_sync(0xffffffffu, ok)) break;
                }
                if (__any_sync(0xffffffffu, wait_step(cr, spins, sleep_ns, kTileMaxSleepNs))) {
                    if (lane == 0) give_up(cr);
#pragma unroll
                    for (int v = 0; v < VEC; ++v) cin[v] = __int_as_float(0x7fc00000);
                    break;
                }
            }
        }
        if (cok && !walk && more) {
            float hend[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) hend[v] = __fmaf_rn(TA[v], cin[v], TB[v]);
            put_states<VEC>(cr.inc + base, hend, cr.epoch);
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) sm.carry[lane][v] = cin[v];
    }
    csync<NW>();
    float PA[VEC], PB[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { PA[v] = 1.f; PB[v] = 0.f; }
#pragma unroll
    for (int w = 0; w < NW - 1; ++w) {
        if (w < warp) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float a = sm.a[w][lane][v], b = sm.b[w][lane][v];
                PB[v] = __fmaf_rn(a, PB[v], b);
                PA[v] *= a;
            }
        }
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) start[v] = __fmaf_rn(PA[v], sm.carry[lane][v], PB[v]);
}

// Shared memory of the strip kernel's carry: every warp's aggregate.
template <int VEC, int NW>
struct StripSmem {
    float a[NW][32][VEC];
    float b[NW][32][VEC];
};

// Whole CTA, strip kernel.  (A, B): this thread's aggregate over its R rows.
// The state before this chunk is `init` (first chunk; every warp passes it) or
// this CTA's state after the previous chunk of the same channel strip,
// carry[par] ([32][VEC] in shared memory, par = chunk parity).  After one
// barrier every warp folds the aggregates of the warps before it, in row
// order, into that state -- the state entering its rows -- and the last warp
// continues with its own aggregate and leaves the state after the chunk in
// carry[par ^ 1].  Every warp applies the same operations in the same order,
// so the bits are fixed by position.  Returns in `start` the state entering
// this thread's first row.
template <int VEC, int NW>
__device__ __forceinline__ void strip_carry(StripSmem<VEC, NW>& sm, const float (&A)[VEC],
                                            const float (&B)[VEC], const float (&init)[VEC],
                                            float (&start)[VEC], float (*carry)[32][VEC], int par,
                                            bool first, bool cok) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        sm.a[warp][lane][v] = A[v];
        sm.b[warp][lane][v] = B[v];
    }
    csync<NW>();
    float st[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) st[v] = first ? (cok ? init[v] : 0.f) : carry[par][lane][v];
#pragma unroll kFoldUnroll
    for (int w = 0; w < warp; ++w)
#pragma unroll
        for (int v = 0; v < VEC; ++v) st[v] = __fmaf_rn(sm.a[w][lane][v], st[v], sm.b[w][lane][v]);
#pragma unroll
    for (int v = 0; v < VEC; ++v) start[v] = st[v];
    if (warp == NW - 1) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) carry[par ^ 1][lane][v] = __fmaf_rn(A[v], st[v], B[v]);
    }
}

// Whole CTA, walker protocol, look-ahead phase: combine the warp aggregates
// of a tile and publish the tile aggregate (no wait, no output).
template <int VEC, int NW>
__device__ __forceinline__ void tile_publish_agg(CarrySmem<VEC, NW>& sm, const float (&A)[VEC],
                                                 const float (&B)[VEC], const Carry& cr,
                                                 const Geom& g, int64_t q, int64_t c, bool cok) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        sm.a[warp][lane][v] = A[v];
        sm.b[warp][lane][v] = B[v];
    }
    csync<NW>();
    if (warp == 0 && cok && q < g.n_chunks - 1) {
        float TA[VEC], TB[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { TA[v] = 1.f; TB[v] = 0.f; }
#pragma unroll
        for (int w = 0; w < NW; ++w)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float a = sm.a[w][lane][v], b = sm.b[w][lane][v];
                TB[v] = __fmaf_rn(a, TB[v], b);
                TA[v] *= a;
            }
#pragma unroll
        for (int v = 0; v < VEC; ++v)
            st_pkt2(cr.agg + 2 * ((c + v) * g.n_chunks + q), pkt(TA[v], cr.epoch),
                    pkt(TB[v], cr.epoch));
    }
    csync<NW>();  // the smem is reused by the next phase
}

}  // namespace lrs
