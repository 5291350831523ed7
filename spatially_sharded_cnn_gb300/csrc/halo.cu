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

// The halo-padded layout of one rank: rows of Wp = Wl + 2 * kHaloCols floats,
// the block's own columns at [kHaloCols, kHaloCols + Wl).  Everything moves in
// 16-byte pieces (kHaloCols = 4, Wl % 4 == 0): Q = Wp / 4 float4s per row.
__global__ void halo_pad_kernel(const float4* __restrict__ x, float4* __restrict__ xp, long long rows, int Q) {
    const long long total = rows * Q;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        const long long r = q / Q;
        const int k = (int)(q - r * Q);
        xp[q] = k > 0 && k < Q - 1 ? __ldg(x + r * (Q - 2) + (k - 1)) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
}
// buf[r] = the first (side 0) or last (side 1) own float4 of row r
__global__ void halo_pack_kernel(const float4* __restrict__ xp, float4* __restrict__ buf, long long rows, int Q,
                                 int side) {
    const int k = side ? Q - 2 : 1;
    for (long long r = blockIdx.x * (long long)blockDim.x + threadIdx.x; r < rows;
         r += (long long)gridDim.x * blockDim.x)
        buf[r] = __ldg(xp + r * Q + k);
}
// the left (side 0) or right (side 1) margin of row r = buf[r], or zeros
__global__ void halo_unpack_kernel(const float4* __restrict__ buf, float4* __restrict__ xp, long long rows, int Q,
                                   int side) {
    const int k = side ? Q - 1 : 0;
    for (long long r = blockIdx.x * (long long)blockDim.x + threadIdx.x; r < rows;
         r += (long long)gridDim.x * blockDim.x)
        xp[r * Q + k] = buf ? __ldg(buf + r) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
}

unsigned grid_for(long long n) {
    const long long b = (n + 255) / 256;
    return (unsigned)(b < 152LL * 32 ? (b > 0 ? b : 1) : 152LL * 32);
}

}  // namespace

hc_status launch_halo_pad(const hc_conv_desc* d, int Wl, const float* x, float* xp, cudaStream_t st) {
    const long long rows = (long long)d->N * d->C_in * d->H;
    const int Q = (Wl + 2 * kHaloCols) / 4;
    halo_pad_kernel<<<grid_for(rows * Q), 256, 0, st>>>(reinterpret_cast<const float4*>(x),
                                                        reinterpret_cast<float4*>(xp), rows, Q);
    return launched("halo_pad_kernel", st);
}

hc_status launch_halo_pack(const hc_conv_desc* d, int Wl, const float* xp, int side, float* buf, cudaStream_t st) {
    const long long rows = (long long)d->N * d->C_in * d->H;
    const int Q = (Wl + 2 * kHaloCols) / 4;
    halo_pack_kernel<<<grid_for(rows), 256, 0, st>>>(reinterpret_cast<const float4*>(xp),
                                                     reinterpret_cast<float4*>(buf), rows, Q, side);
    return launched("halo_pack_kernel", st);
}

hc_status launch_halo_unpack(const hc_conv_desc* d, int Wl, const float* buf, int side, float* xp, cudaStream_t st) {
    const long long rows = (long long)d->N * d->C_in * d->H;
    const int Q = (Wl + 2 * kHaloCols) / 4;
    halo_unpack_kernel<<<grid_for(rows), 256, 0, st>>>(reinterpret_cast<const float4*>(buf),
                                                       reinterpret_cast<float4*>(xp), rows, Q, side);
    return launched("halo_unpack_kernel", st);
}

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
