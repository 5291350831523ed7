// halo.cu -- explicit halo exchange + concat (kwkr.cn news/18980 section 2.2,
// steps 1-2; NVIDIA blog "Perception model training for autonomous vehicles
// with tensor parallelism", Figure 1).  Shard r's extended tile is the left
// neighbour's last halo_left columns, its own block, and the right
// neighbour's first halo_right columns; columns past the image edge are zero.
#include "common.cuh"

namespace hc {
namespace {

struct HaloTab {
    int hl[kMaxKernelShards];
    int hr[kMaxKernelShards];
};

// One thread per float of x_ext [S][N][C][H][We]; consecutive threads walk
// consecutive columns, so reads and writes are coalesced.
__global__ void halo_gather_kernel(const float* __restrict__ x, float* __restrict__ xe, long long rows_per_shard,
                                   int W, int Wl, int We, long long total, HaloTab tab) {
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(q % We);
        const long long row = q / We;              // (r, n, c, h)
        const int r = (int)(row / rows_per_shard);
        const long long src_row = row - r * rows_per_shard;  // (n, c, h)
        const int hl = tab.hl[r], hr = tab.hr[r];
        const int col = r * Wl - hl + t;
        float v = 0.0f;
        if (t < hl + Wl + hr && col >= 0 && col < W) v = __ldg(x + src_row * W + col);
        xe[q] = v;
    }
}

}  // namespace

hc_status launch_halo_gather(const hc_conv_desc* d, const Plan& p, const float* x, float* x_ext, cudaStream_t st) {
    HaloTab tab;
    for (int r = 0; r < p.S; r++) {
        tab.hl[r] = p.ext[r].halo_left;
        tab.hr[r] = p.ext[r].halo_right;
    }
    const long long rows = (long long)d->N * d->C_in * d->H;
    const long long total = rows * p.S * p.We;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    const unsigned grid = (unsigned)(blocks < 152LL * 64 ? blocks : 152LL * 64);
    halo_gather_kernel<<<grid, threads, 0, st>>>(x, x_ext, rows, d->W, p.Wl, p.We, total, tab);
    return launched();
}

}  // namespace hc
