// lr_common.cuh -- device machinery shared by every chunked-scan kernel:
// storage packs (fp32 / bf16, 16-byte vectors), the tile ticket, and the
// single-pass decoupled look-back that carries the recurrence state across
// time chunks.
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
//     owns channels [l*VEC, l*VEC+VEC) of the tile (one 16-byte vector per row,
//     so one warp row is a 512-byte coalesced segment), warp w owns the R
//     consecutive rows [w*R, w*R+R) in scan order;
//   * each thread scans its R rows sequentially in registers (depth R), the
//     NW warp aggregates are combined through shared memory (depth NW), and the
//     tiles along time are chained by decoupled look-back over a window of 32
//     predecessors at a time (depth ~ number of tiles / 32 in the worst case,
//     one step in the common case), so a million-step sequence is one launch;
//   * tiles are handed out by an atomic ticket in scan order, so every tile a
//     CTA waits for belongs to a CTA that is already running: the wait always
//     ends.  Every wait is still bounded (spin_limit polls); when it runs out
//     the tile records LR_ERR_TIMEOUT in the error word, publishes NaN and
//     finishes, so its successors do not wait in turn.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lrs {

constexpr uint32_t ST_X = 0;    // nothing published (or an older launch's flag)
constexpr uint32_t ST_AGG = 1;  // tile aggregate (A, B) published
constexpr uint32_t ST_INC = 2;  // inclusive state at the tile's last row published
constexpr uint32_t ERRBIT_TIMEOUT = 1u;

// Look-back descriptors: one flag word and 3*CW floats per tile.  A flag is
// (epoch << 2) | state; a flag whose epoch differs from this launch's is read
// as ST_X, so the descriptors never need clearing between launches.
struct Lookback {
    uint32_t* flags;     // [n_tiles]
    float* agg_a;        // [n_tiles * CW]  product of a over the tile
    float* agg_b;        // [n_tiles * CW]  state after the tile from zero
    float* inc;          // [n_tiles * CW]  state after the tile (true carry)
    uint32_t* ticket;    // tile ticket counter (0 between launches)
    uint32_t* err;       // sticky error bits
    uint32_t epoch;      // 1 .. 2^30-1
    uint32_t spin_limit; // polls before a wait gives up
};

struct Geom {
    int64_t T;            // rows
    int64_t C;            // channels (B*D)
    int64_t D;            // features (per-feature parameters use c % D)
    int64_t n_chunks;     // ceil(T / L)
    int n_ct;             // ceil(C / CW)
    uint32_t n_launch;    // CTAs launched (= tiles; the timeout test launches fewer)
    uint32_t ticket_base; // first ticket value mapped to tile 0 + ticket_base
};

// ------------------------------------------------------------- memory ops

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Streaming 16-byte loads of read-once inputs (no L1 allocation).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ void st_u4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
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
// the vector path and one element on the scalar path.

template <typename S, int VEC>
struct Pack;

template <int VEC>
struct Pack<float, VEC> {
    static_assert(VEC == 4 || VEC == 1, "fp32 packs hold 4 or 1 elements");
    float v[VEC];
    __device__ __forceinline__ void load(const float* p) {
        if constexpr (VEC == 4) {
            uint4 r = ld_stream_u4(p);
            v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
            v[2] = __uint_as_float(r.z); v[3] = __uint_as_float(r.w);
        } else {
            v[0] = __ldg(p);
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
    static_assert(VEC == 8 || VEC == 1, "bf16 packs hold 8 or 1 elements");
    static constexpr int NW_ = VEC == 8 ? 4 : 1;
    uint32_t w[NW_];
    __device__ __forceinline__ void load(const __nv_bfloat16* p) {
        if constexpr (VEC == 8) {
            uint4 r = ld_stream_u4(p);
            w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
        } else {
            w[0] = (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p));
        }
    }
    __device__ __forceinline__ float get(int i) const {
        if constexpr (VEC == 8) return (i & 1) ? bf_hi(w[i >> 1]) : bf_lo(w[i >> 1]);
        else return bf_lo(w[0]);
    }
    __device__ __forceinline__ void ident(float x) {
        uint32_t b = bf_bits(x);
#pragma unroll
        for (int i = 0; i < NW_; ++i) w[i] = VEC == 8 ? (b | (b << 16)) : b;
    }
};

// Store VEC fp32 values to storage type S (bf16: round to nearest-even).
template <typename S, int VEC>
__device__ __forceinline__ void store_vec(S* p, const float (&x)[VEC]) {
    if constexpr (sizeof(S) == 4) {
        if constexpr (VEC == 4)
            st_u4(p, make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]),
                                __float_as_uint(x[2]), __float_as_uint(x[3])));
        else
            *reinterpret_cast<float*>(p) = x[0];
    } else {
        if constexpr (VEC == 8)
            st_u4(p, make_uint4(bf_pack(x[0], x[1]), bf_pack(x[2], x[3]), bf_pack(x[4], x[5]),
                                bf_pack(x[6], x[7])));
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

// Descriptor payload: VEC floats per lane, L2 only (.cg) so no stale L1 line
// from an earlier launch is ever read.
template <int VEC>
__device__ __forceinline__ void put_payload(float* p, const float (&x)[VEC]) {
    if constexpr (VEC % 4 == 0) {
#pragma unroll
        for (int i = 0; i < VEC; i += 4)
            __stcg(reinterpret_cast<float4*>(p + i), make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]));
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) __stcg(p + i, x[i]);
    }
}
template <int VEC>
__device__ __forceinline__ void get_payload(const float* p, float (&x)[VEC]) {
    if constexpr (VEC % 4 == 0) {
#pragma unroll
        for (int i = 0; i < VEC; i += 4) {
            float4 f = __ldcg(reinterpret_cast<const float4*>(p + i));
            x[i] = f.x; x[i + 1] = f.y; x[i + 2] = f.z; x[i + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) x[i] = __ldcg(p + i);
    }
}

// ------------------------------------------------------------ the ticket

// Returns this CTA's tile number (in scan order).  The CTA that draws the last
// ticket of the launch resets the counter for the next launch on the stream.
__device__ __forceinline__ uint32_t take_ticket(const Lookback& lb, const Geom& g) {
    __shared__ uint32_t s_ticket;
    if (threadIdx.x == 0) {
        uint32_t t = atomicAdd(lb.ticket, 1u);
        if (t == g.n_launch - 1) atomicExch(lb.ticket, 0u);
        s_ticket = t + g.ticket_base;
    }
    __syncthreads();
    return s_ticket;
}

// ---------------------------------------------------------- publication

// Whole warp: write this lane's payload, then lane 0 raises the flag.
template <int VEC>
__device__ __forceinline__ void publish(float* payload, const float (&x)[VEC], uint32_t* flag,
                                        uint32_t word) {
    put_payload<VEC>(payload, x);
    __threadfence();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) st_release_u32(flag, word);
}

// Whole warp: the carry entering scan-order chunk q (q >= 1) for channel tile
// j, i.e. the state after chunk q-1.  Walks back over windows of 32
// predecessors (lane i watches chunk base-i) until the nearest chunk p whose
// inclusive state is visible, with every chunk between p and q-1 showing its
// aggregate.  The carry is then rebuilt by folding forward, oldest first:
//     h = INC(p);  h = A(i) h + B(i)  for i = p+1 .. q-1,
// which is exactly the fused multiply-add each of those chunks performs when
// it publishes its own inclusive state.  The result is therefore bitwise the
// same whichever p the race happened to expose: the scan is deterministic.
// Returns false (carry = NaN, error bit set) when the wait ran out.
template <int VEC, int CW>
__device__ bool lookback(const Lookback& lb, int64_t q, int j, int n_ct, float (&cin)[VEC]) {
    const int lane = threadIdx.x & 31;
    int64_t base = q - 1;
    int64_t first = -1;  // nearest chunk with a visible inclusive state
    uint32_t spins = 0;
    uint32_t sleep_ns = 0;
    while (first < 0) {
        const int64_t pred = base - lane;
        uint32_t st = ST_X;
        if (pred >= 0) {
            const uint32_t f = ld_acquire_u32(lb.flags + pred * n_ct + j);
            if ((f >> 2) == lb.epoch) st = f & 3u;
        }
        const unsigned inc = __ballot_sync(0xffffffffu, pred >= 0 && st == ST_INC);
        const unsigned ok = __ballot_sync(0xffffffffu, pred < 0 || st != ST_X);
        if (inc) {
            const int p = __ffs(inc) - 1;
            const unsigned need = p == 31 ? 0xffffffffu : ((2u << p) - 1u);
            if ((ok & need) == need) { first = base - p; break; }
        } else if (ok == 0xffffffffu) {
            base -= 32;  // 32 aggregates, no inclusive state yet: look further back
            continue;
        }
        ++spins;
        bool give_up = spins > lb.spin_limit;
        if ((spins & 63u) == 0 && (ld_relaxed_u32(lb.err) & ERRBIT_TIMEOUT)) give_up = true;
        if (__any_sync(0xffffffffu, give_up)) {
            if (lane == 0) atomicOr(lb.err, ERRBIT_TIMEOUT);
#pragma unroll
            for (int v = 0; v < VEC; ++v) cin[v] = __int_as_float(0x7fc00000);
            return false;
        }
        if (sleep_ns) __nanosleep(sleep_ns);
        sleep_ns = sleep_ns == 0 ? 32 : (sleep_ns < 1024 ? sleep_ns * 2 : 1024);
    }
    __syncwarp();
    float h[VEC];
    get_payload<VEC>(lb.inc + (first * n_ct + j) * CW + lane * VEC, h);
#pragma unroll 4
    for (int64_t i = first + 1; i < q; ++i) {
        const int64_t tile = i * n_ct + j;
        float pa[VEC], pb[VEC];
        get_payload<VEC>(lb.agg_a + tile * CW + lane * VEC, pa);
        get_payload<VEC>(lb.agg_b + tile * CW + lane * VEC, pb);
#pragma unroll
        for (int v = 0; v < VEC; ++v) h[v] = __fmaf_rn(pa[v], h[v], pb[v]);
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) cin[v] = h[v];
    return true;
}

// Shared memory for combining the NW warp aggregates of a tile.
template <int VEC, int NW>
struct CarrySmem {
    float a[NW][32][VEC];
    float b[NW][32][VEC];
    float carry[32][VEC];
};

// Whole CTA.  (A, B): this thread's aggregate over its R rows (scan order).
// init: state before the whole scan (used by warp 0 when q == 0).
// Returns in `start` the state entering this thread's first row.
template <int VEC, int NW>
__device__ __forceinline__ void tile_carry(CarrySmem<VEC, NW>& sm, const float (&A)[VEC],
                                           const float (&B)[VEC], const float (&init)[VEC],
                                           float (&start)[VEC], const Lookback& lb, int64_t q,
                                           int j, int n_ct) {
    constexpr int CW = 32 * VEC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        sm.a[warp][lane][v] = A[v];
        sm.b[warp][lane][v] = B[v];
    }
    __syncthreads();
    if (warp == 0) {
        float TA[VEC], TB[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { TA[v] = 1.f; TB[v] = 0.f; }
#pragma unroll
        for (int w = 0; w < NW; ++w)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float a = sm.a[w][lane][v], b = sm.b[w][lane][v];
                TB[v] = a * TB[v] + b;
                TA[v] *= a;
            }
        const int64_t tile = q * n_ct + j;
        float cin[VEC];
        if (q == 0) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) cin[v] = init[v];
        } else {
            put_payload<VEC>(lb.agg_a + tile * CW + lane * VEC, TA);
            publish<VEC>(lb.agg_b + tile * CW + lane * VEC, TB, lb.flags + tile,
                         (lb.epoch << 2) | ST_AGG);
            lookback<VEC, CW>(lb, q, j, n_ct, cin);
        }
        float hend[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) hend[v] = __fmaf_rn(TA[v], cin[v], TB[v]);
        publish<VEC>(lb.inc + tile * CW + lane * VEC, hend, lb.flags + tile, (lb.epoch << 2) | ST_INC);
#pragma unroll
        for (int v = 0; v < VEC; ++v) sm.carry[lane][v] = cin[v];
    }
    __syncthreads();
    float PA[VEC], PB[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { PA[v] = 1.f; PB[v] = 0.f; }
#pragma unroll
    for (int w = 0; w < NW - 1; ++w) {
        if (w < warp) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float a = sm.a[w][lane][v], b = sm.b[w][lane][v];
                PB[v] = a * PB[v] + b;
                PA[v] *= a;
            }
        }
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) start[v] = __fmaf_rn(PA[v], sm.carry[lane][v], PB[v]);
}

}  // namespace lrs
