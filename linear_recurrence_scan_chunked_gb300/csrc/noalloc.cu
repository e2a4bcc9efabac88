// noalloc.cu -- lr_scan_fwd_noalloc: the forward scan for callers that must
// not allocate device memory.
//
// Who needs it: code that runs under someone else's memory manager -- an
// inference engine or framework plugin that owns every device byte and plans
// its budget ahead, a latency-critical server loop.  lr_scan_fwd grows a
// cached workspace with cudaMalloc on first use (and cudaFree + cudaMalloc
// when a larger problem arrives); a hidden allocation can fail at run time,
// fragments the owner's pool, and cudaFree synchronises the whole device.
// This variant keeps its scratch (the chunk-state packets and the tile
// ticket) in one fixed, file-scope __device__ array instead, so it calls
// no cudaMalloc, cudaFree or allocating library routine.
//
// Costs and rules of the fixed array:
//   * every GPU that loads the library holds kScratchBytes (8 MiB) of device
//     memory until the process exits;
//   * problems needing more carry packets than fit are rejected with
//     LR_ERR_TOO_LARGE: ~1 M 8-byte packets, one per channel per chunk of
//     time steps (the chain protocol), two (look-back protocol, short
//     problems) or three (walker protocol, long ones); the cluster kernel's
//     problems (at most 2048 steps) need none;
//   * every call shares the one array: two calls whose kernels overlap on the
//     GPU (different streams, no ordering between them) race on it and give
//     wrong results.  Order such calls on one stream or with events.
//   * the array keeps the last call's contents.  Packets are tagged with the
//     launch's epoch, which the kernels take from the array's ticket word on
//     the device, so packets of earlier calls are ignored; before every
//     launch one 8-byte memset (not an allocation) clears the internal error
//     word and the tile counter, and leaves the epoch alone.
//   * the first call on a device looks up the array's device address with
//     cudaGetSymbolAddress (host code cannot use the symbol itself); make that
//     first call before any stream capture.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "lr_launch.h"
#include "lrscan.h"

namespace {

using namespace lrs;

constexpr size_t kScratchBytes = size_t(8) << 20;
// Header: bytes 4..7 the internal error word, 8..15 the 64-bit ticket word
// (bytes 8..11 the tile counter, 12..15 the last retired epoch); packets from
// byte 256 on.  Bytes 4..11 are cleared before every launch.
constexpr size_t kHeaderBytes = 256;
constexpr size_t kErrOff = 4, kTicketOff = 8;
constexpr uint32_t kSpinLimit = 1u << 21;
constexpr int kMaxDevices = 64;
// Launches after which the packets and the epoch are cleared (the device's
// epochs never wrap into packets of earlier calls).
constexpr uint64_t kEpochClear = 1ull << 31;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct NoAllocDev {
    unsigned char* base = nullptr;  // device address of g_scratch on this device
    uint64_t launches = 0;          // launches since the last clear
};
std::mutex g_na_mu;
NoAllocDev g_na[kMaxDevices];

}  // namespace

extern "C" int lr_scan_fwd_noalloc(const void* a, const void* b, const void* h0, void* h,
                                   int64_t B, int64_t T, int64_t D, int dtype,
                                   uint32_t* err_dev, void* stream) {
    if (dtype != LR_F32 && dtype != LR_BF16) return LR_ERR_INVALID_ARG;
    if (B < 0 || T < 0 || D < 0) return LR_ERR_INVALID_ARG;
    if (B == 0 || T == 0 || D == 0) return LR_OK;
    const int64_t lim = (int64_t)1 << 62;
    if (B > lim / T || B * T > lim / D) return LR_ERR_TOO_LARGE;
    if (!a || !b || !h) return LR_ERR_INVALID_ARG;
    const size_t es = dtype == LR_BF16 ? 2 : 4;
    bool vec = (D % kvec(dtype, true)) == 0;
    for (const void* p : {a, b, (const void*)h, h0}) {
        if (!p) continue;
        if ((uintptr_t)p % es) return LR_ERR_ALIGN;
        vec = vec && ((uintptr_t)p % 16 == 0);
    }
    if (err_dev && ((uintptr_t)err_dev % 4)) return LR_ERR_ALIGN;

    const int64_t C = B * D;
    const CarryPlan cp = carry_plan(OP_SCAN_FWD, dtype, vec, use_tma(dtype, vec, T, C), T, C);
    const TileShape ts = cp.ts;
    const int64_t n_chunks = cp.n_chunks;
    const int64_t n_ct = (C + ts.CW - 1) / ts.CW;
    if (n_ct > INT32_MAX || n_chunks > INT32_MAX / 4 / n_ct) return LR_ERR_TOO_LARGE;
    const size_t tiles = (size_t)(n_chunks * n_ct);
    const size_t pk_bytes = (cp.inc_elems + cp.agg_elems) * sizeof(u64);
    if (kHeaderBytes + pk_bytes > kScratchBytes) return LR_ERR_TOO_LARGE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LR_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    std::lock_guard<std::mutex> lock(g_na_mu);
    NoAllocDev& nd = g_na[dev];
    if (!nd.base) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return LR_ERR_CUDA;
        nd.base = (unsigned char*)p;
    }
    u64* pk = (u64*)(nd.base + kHeaderBytes);
    if (++nd.launches >= kEpochClear) {  // forget every old packet; epochs restart at 1
        nd.launches = 1;
        if (cudaMemsetAsync(nd.base, 0, kScratchBytes, s) != cudaSuccess) return LR_ERR_CUDA;
    }
    // the internal error word and the tile counter (a launch that gave up
    // may have left it mid-count); not the epoch
    if (cudaMemsetAsync(nd.base + kErrOff, 0, 8, s) != cudaSuccess) return LR_ERR_CUDA;

    Geom g;
    g.T = T;
    g.C = C;
    g.D = D;
    set_channel_div(g);
    g.n_chunks = n_chunks;
    g.n_ct = (int)n_ct;
    g.n_tiles = (uint32_t)tiles;
    g.n_draws = 0;
    g.ticket_base = 0;
    g.max_grid = 0;
    Carry cr;
    cr.inc = pk;
    cr.agg = pk + cp.inc_elems;
    cr.tk = (u64*)(nd.base + kTicketOff);
    cr.err = err_dev ? err_dev : (uint32_t*)(nd.base + kErrOff);
    cr.epoch = 0;  // taken on the device from the ticket word
    cr.spin_limit = kSpinLimit;
    cr.mode = cp.mode;
    cr.n_walk = cp.n_walk;
    cr.wv = cp.wv;
    cr.tma = cp.tma ? 1 : 0;
    if (launch_scan_fwd(dtype, vec, a, b, h0, h, g, cr, s) != cudaSuccess) return LR_ERR_CUDA;
    return LR_OK;
}
