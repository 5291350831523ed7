// halo.cu -- explicit halo exchange + concat (kwkr.cn news/18980 section 2.2,
// steps 1-2; NVIDIA blog "Perception model training for autonomous vehicles
// with tensor parallelism", Figure 1).  Shard r's extended tile is the left
// neighbour's last halo_left columns, its own block, and the right
// neighbour's first halo_right columns; columns past the image edge are zero.
// With row shards too (kwkr.cn 5.2, Shard(2)) the tile also takes the halo
// rows above and below its block, and the shards form a row x column grid.
#include "common.cuh"

namespace hc {
namespace {

struct HaloTab {
    int hl[kMaxKernelShards];  // per column shard: halo columns left / right
    int hr[kMaxKernelShards];
    int ht[kMaxKernelShards];  // per row shard: halo rows above / below
    int hb[kMaxKernelShards];
};

// One thread per float of x_ext [Q][N][C][He][We], shard q = a * S + b (row
// block a, column block b); consecutive threads walk consecutive columns, so
// reads and writes are coalesced.
__global__ void halo_gather_kernel(const float* __restrict__ x, float* __restrict__ xe, long long planes, int H,
                                   int W, int Hl, int Wl, int He, int We, int S, long long total, HaloTab tab) {
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(q % We);
        long long rest = q / We;
        const int rr = (int)(rest % He);
        rest /= He;
        const long long plane = rest % planes;  // (n, c)
        const int qq = (int)(rest / planes);
        const int a = qq / S, b = qq - a * S;
        const int hl = tab.hl[b], hr = tab.hr[b], ht = tab.ht[a], hb = tab.hb[a];
        const int col = b * Wl - hl + t, row = a * Hl - ht + rr;
        float v = 0.0f;
        if (t < hl + Wl + hr && rr < ht + Hl + hb && col >= 0 && col < W && row >= 0 && row < H)
            v = __ldg(x + (plane * H + row) * W + col);
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
    for (int a = 0; a < p.Sh; a++) {
        tab.ht[a] = p.ext_h[a].halo_left;
        tab.hb[a] = p.ext_h[a].halo_right;
    }
    const long long planes = (long long)d->N * d->C_in;
    const long long total = planes * p.Q * p.He * p.We;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    const unsigned grid = (unsigned)(blocks < 152LL * 64 ? blocks : 152LL * 64);
    halo_gather_kernel<<<grid, threads, 0, st>>>(x, x_ext, planes, d->H, d->W, p.Hl, p.Wl, p.He, p.We, p.S, total,
                                                 tab);
    return launched("halo_gather_kernel", st);
}

}  // namespace hc
