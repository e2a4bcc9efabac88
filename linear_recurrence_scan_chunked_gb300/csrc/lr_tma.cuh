// lr_tma.cuh -- tile staging with the Tensor Memory Accelerator (sm_100+).
//
// A tile of every input array (L time rows x CW channels of the [T, C]
// sequence, C = B*D contiguous) is one 2-D box of a tensor map: one
// cp.async.bulk.tensor per array per tile moves it from HBM into a stage of a
// shared-memory ring, and an mbarrier counts its bytes in.  One thread (or, in
// the TMA chain kernel, a producer warp) keeps the ring's stages in flight per
// CTA without holding registers, so the bytes in flight per SM no longer depend
// on the registers of the arithmetic warps (in the register-double-buffered
// kernels they do).
//
// Shared-memory layout of one stage: array k of the operation at byte offset
// tma_off<Op>(k) (128-byte aligned), rows in time order, row pitch CW *
// sizeof(S) (512 B fp32, 256 B bf16).  Lane l of a warp reads its VEC
// channels of a row at byte l * VEC * sizeof(S): a warp reads one whole row,
// conflict free.
//
// An operation that supports TMA staging provides
//   TMA_N                    input arrays staged per tile
//   tma_shift(k)             first time row of array k relative to the chunk's
//                            first row (0, or -1 for h_{t-1} / c_{t-1} / y_{t-1})
//   tma_extra(k)             rows beyond L (1 when the shifted array also needs
//                            the chunk's last row)
//   tma_arrays(p, ptr)       the device pointer of each array (nullptr: not
//                            staged this launch, the op does not read it)
#pragma once

#include <cuda.h>

#include "lr_common.cuh"

namespace lrs {

constexpr int TMA_MAX_ARR = 6;

// Tensor maps of one launch (kernel parameter, __grid_constant__).
struct TmaDesc {
    CUtensorMap map[TMA_MAX_ARR];
    uint32_t present;   // bit k: array k is staged
    uint32_t tx_bytes;  // bytes one stage receives
};

// Host: 2-D tensor map over the [T, C] sequence at ptr (dtype 0 fp32, 1 bf16)
// with a box of box_rows x box_c elements, zero fill outside.  False when the
// driver refuses it.
bool tma_encode(CUtensorMap* m, const void* ptr, int dtype, int64_t T, int64_t C, int box_c,
                int box_rows);

template <class Op>
__host__ __device__ constexpr uint32_t tma_arr_bytes(int k) {
    return (uint32_t)(Op::NW * Op::R + Op::tma_extra(k)) * 32u * Op::VEC *
           (uint32_t)sizeof(typename Op::S);
}
template <class Op>
__host__ __device__ constexpr uint32_t tma_off(int k) {
    uint32_t o = 0;
    for (int j = 0; j < k; ++j) o += (tma_arr_bytes<Op>(j) + 127u) & ~127u;
    return o;
}
template <class Op>
__host__ __device__ constexpr uint32_t tma_stage_bytes() {
    return tma_off<Op>(Op::TMA_N);
}

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
// Make the barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* b, uint32_t tx) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)),
                 "r"(tx)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// As mbar_try_wait, acquiring at cluster scope: the phase completes on data
// that other CTAs of the cluster stored into this CTA's shared memory.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait for the phase of parity `parity` of barrier b to complete.
// Returns false when it gave up (about kMbarLimitNs, or the launch's sticky
// error word says another CTA already gave up).
constexpr uint64_t kMbarLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, const uint32_t* err) {
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(b, parity)) return true;
        if ((n & 255u) == 0) {
            if (globaltimer_ns() - t0 > kMbarLimitNs) return false;
            if (ld_relaxed_u32(err) & ERRBIT_TIMEOUT) return false;
        }
    }
}
// One 2-D box {x: channel, y: time row} of tensor map m into shared memory,
// completing on barrier b.  x is a multiple of CW (16-byte aligned); y may be
// -1 or past the end (those rows are zero-filled; the ops never read them).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, int32_t x, int32_t y,
                                            uint64_t* b) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(b))
        : "memory");
}

// Bring a tensor map (a __grid_constant__ kernel parameter) into the
// descriptor cache ahead of its first copy.
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// As tma_load_2d, with an L2 eviction-priority policy (createpolicy) for the
// lines it reads.
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* m, int32_t x,
                                                 int32_t y, uint64_t* b, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(b)), "l"(pol)
        : "memory");
}

// ---------------------------------------------------------- clusters
// This CTA's rank in its thread-block cluster and the cluster's CTA count.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_ctas() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// The cluster barrier, split: every thread of every CTA arrives, then waits.
// The relaxed arrive orders no memory access of its own (a barrier's
// initialisation is published by fence.mbarrier_init before it); the wait
// acquires.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address that `p` (in this CTA's shared memory) has in CTA `rank` of
// the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    return a;
}
// An asynchronous store of two floats into another CTA's shared memory
// (cluster addresses from cluster_map) that counts its 8 bytes on that CTA's
// barrier `bar`: the storing thread does not wait for it.
__device__ __forceinline__ void st_async_f2(uint32_t dst, float x, float y, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(dst),
                 "f"(x), "f"(y), "r"(bar)
                 : "memory");
}
// As st_async_f2, four floats (16 bytes, 16-byte aligned).
__device__ __forceinline__ void st_async_f4(uint32_t dst, float x, float y, float z, float w,
                                            uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(dst),
        "f"(x), "f"(y), "f"(z), "f"(w), "r"(bar)
        : "memory");
}

// ---------------------------------------------------------- tile sources
// Where Op::load takes the rows of its arrays from: global memory (register
// kernels) or the staged tile in shared memory (TMA kernels).

struct GlobalSrc {
    int64_t C;  // row pitch in elements
    int64_t c;  // first channel of this lane
    template <class P, typename S>
    __device__ __forceinline__ void ld(P& pk, int, const S* base, int64_t t) const {
        pk.load(base + t * C + c);
    }
};

// Global loads carrying an L2 eviction-priority policy.
struct GlobalSrcHint {
    int64_t C;
    int64_t c;
    uint64_t pol;
    template <class P, typename S>
    __device__ __forceinline__ void ld(P& pk, int, const S* base, int64_t t) const {
        pk.load_hint(base + t * C + c, pol);
    }
};

template <class Op>
struct SmemSrc {
    const unsigned char* stage;
    int64_t row0;  // time of the chunk's first row
    int lane_e;    // lane * VEC
    template <class P, typename S>
    __device__ __forceinline__ void ld(P& pk, int k, const S*, int64_t t) const {
        constexpr int CW = 32 * Op::VEC;
        const int row = (int)(t - row0) - Op::tma_shift(k);
        pk.load_shared(reinterpret_cast<const S*>(stage + tma_off<Op>(k)) + row * CW + lane_e);
    }
};

}  // namespace lrs
