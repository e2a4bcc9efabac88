// lr_launch.h -- host-side interface between the C ABI (lr_api.cu) and the
// kernel translation units.  Each operation exposes its tile shape (so the
// API can size the look-back workspace) and a launcher that picks the
// template instance for the storage type and the vector / scalar path.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lr_common.cuh"

namespace lrs {

struct TileShape {
    int L;    // time rows per tile
    int CW;   // channels per tile
    int threads;
};

enum Op { OP_SCAN_FWD = 0, OP_SCAN_BWD, OP_SRU_FWD, OP_SRU_BWD, OP_DEER, OP_COUNT };

// Launch configuration of every kernel: NW warps per CTA, R rows per thread
// (tile = NW*R rows), VEC channels per lane (16-byte vectors on the vector
// path, one element on the scalar path).  One table, used both to instantiate
// the kernels and to size the workspace.
struct KCfg {
    int NW;
    int R;
};
constexpr KCfg kcfg(Op op, int dtype) {
    return op == OP_SCAN_FWD ? KCfg{8, dtype == 1 ? 4 : 8}
         : op == OP_SCAN_BWD ? KCfg{8, dtype == 1 ? 2 : 4}
         : op == OP_SRU_FWD  ? KCfg{8, dtype == 1 ? 2 : 4}
         : op == OP_SRU_BWD  ? KCfg{8, dtype == 1 ? 2 : 4}
         :                     KCfg{8, dtype == 1 ? 2 : 4};
}
constexpr int kvec(int dtype, bool vec) { return vec ? (dtype == 1 ? 8 : 4) : 1; }

inline TileShape tile_shape(Op op, int dtype, bool vec) {
    const KCfg k = kcfg(op, dtype);
    return TileShape{k.NW * k.R, 32 * kvec(dtype, vec), 32 * k.NW};
}

cudaError_t launch_scan_fwd(int dtype, bool vec, const void* a, const void* b, const void* h0,
                            void* h, const Geom& g, const Lookback& lb, cudaStream_t s);

cudaError_t launch_scan_bwd(int dtype, bool vec, const void* a, const void* h, const void* h0,
                            const void* dh, void* da, void* db, void* dh0, const Geom& g,
                            const Lookback& lb, cudaStream_t s);

cudaError_t launch_sru_fwd(int dtype, bool vec, const void* xt, const void* uf, const void* ur,
                           const void* x, const float* bf, const float* br, const void* c0,
                           void* h, void* c, const Geom& g, const Lookback& lb, cudaStream_t s);

// partials: [n_chunks, C] x 2 (forget, reset) fp32 scratch
cudaError_t launch_sru_bwd(int dtype, bool vec, const void* xt, const void* uf, const void* ur,
                           const void* x, const float* bf, const float* br, const void* c0,
                           const void* c, const void* dh, void* dxt, void* duf, void* dur,
                           void* dx, void* dc0, float* partials, const Geom& g,
                           const Lookback& lb, cudaStream_t s);

cudaError_t launch_bias_reduce(const float* partials, int64_t n_chunks, int64_t B, int64_t D,
                               float* dbf, float* dbr, cudaStream_t s);

// resid: one fp32 slot (as bits), zeroed before the launch, receives max|ynew-yold|
cudaError_t launch_deer_iter(int dtype, bool vec, const float* w, const void* u, const void* h0,
                             const void* yold, void* ynew, uint32_t* resid, const Geom& g,
                             const Lookback& lb, cudaStream_t s);

}  // namespace lrs
