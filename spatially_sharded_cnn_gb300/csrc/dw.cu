// dw.cu -- depthwise K x K convolution (groups = C, stride 1, padding (K-1)/2),
// the ConvNeXt depthwise layer the pages single out for the halo exchange
// (kwkr.cn news/18980 sections 3.2 and 6.2).
//
// Work items.  An item is one (n, c) plane x one 128-column tile of it.  Tiles
// never straddle a shard, so a tile at a shard edge reads its halo columns from
// the neighbouring shard's block (the halo exchange of NVIDIA blog "Perception
// model training for autonomous vehicles with tensor parallelism", Figure 1)
// and zeros past the image edge; only the tile's own 128 columns are written
// (the crop).  Every CTA takes one contiguous range of items.  The forward
// orders them (c, n, column tile), so a tile's horizontal neighbours run just
// before and after it and its halo columns are L2 hits; the backward orders
// them (c, column tile, n), so the weight gradient of one (c, column tile)
// accumulates in registers across consecutive images.
//
// Kernels are persistent (a fixed number of CTAs per SM).  One thread streams the tiles in with
// TMA (a 3-D box of rows h0-P .. h0+TH+P-1 and columns c0-4 .. c0+131 of one
// plane; the box start is 16-byte aligned and out-of-image parts are
// zero-filled by the copy engine) into a ring of shared-memory buffers guarded
// by mbarriers (three stages forward, two backward).  In the forward pass the
// warps run through the jobs independently and the last warp done with a stage
// refills it; in the backward pass a CTA barrier ends each job and one thread
// then refills the stage.  A warp that changes channel reads the weights from global memory.
// Every barrier wait is bounded: a CTA that gives up records HC_ERR_TIMEOUT in
// a status word (read by hc_sync_check), waits for its own copies still in
// flight, and returns.
//
// Each thread computes an 8-row x 4-column block: per input row it reads 12
// floats (three 16-byte shared loads) and issues up to 7 * 4 * K FMAs with the
// plane's K*K weights in registers.
//
// Backward (one kernel, two 8-warp CTAs per SM, 32-row jobs, each CTA on its own
// ring, so one CTA's warps keep the SM busy while the other's wait at their
// per-job barrier; both roles cover the same 8-row blocks of each staged tile):
//   warps 0-3   grad_input = the same stencil over the grad_output tile with the
//               kernel flipped (gx[h][c] = sum_{u,v} w[K-1-u][K-1-v] gy[h+u-P][c+v-P]),
//               plus, in a separate instantiation, a residual gradient;
//   warps 4-7   weight / bias gradients of the block's own grad_output elements,
//               gw[u][v] += gy[h][c] * x[h+u-P][c+v-P], accumulated in registers over
//               all consecutive items of the same (c, column tile) and then reduced
//               across these warps (warp shuffles, then the per-warp sums in warp
//               order) into one partial per run.
// dw_shard_partials_kernel then sums the partials of each (shard, c) in a
// fixed order: the per-shard _Partial gradients.
#include "common.cuh"

namespace hc {
namespace {

constexpr int TW = 128;        // tile width (columns)
constexpr int SMW = TW + 8;    // staged row: 4 halo columns on each side
constexpr int FWD_WARPS = 8;   // forward: 64-row tiles, two CTAs per SM
constexpr int FWD_CTAS = 2;
constexpr int BWD_WARPS = 4;   // backward: 32-row tiles, two CTAs per SM, 4 grad_input + 4 weight-gradient warps each
constexpr int BWD_CTAS = 2;
constexpr int BWD_NSTAGE = 2;  // depth of the backward's ring (two 41.5 KB stages: three would not fit twice per SM)
constexpr int NSTAGE = 3;      // depth of the forward's ring
constexpr int WSLOT = 64;      // floats per warp in the weight-gradient reduction buffer (K*K + bias)
constexpr long long kWaitCycles = 4000000000LL;  // about 2 s at 2 GHz

__device__ int g_dw_status;

template <int K, int WARPS>
struct Geo {
    static constexpr int P = (K - 1) / 2;
    static constexpr int TH = 8 * WARPS;                           // rows per tile
    static constexpr int R = TH + 2 * P;                           // staged rows
    static constexpr int TILE = ((R * SMW + 31) / 32) * 32;        // floats per buffer (128-byte multiple)
    static constexpr unsigned BYTES = (unsigned)(R * SMW * 4);     // bytes one TMA box delivers
};

// ---- mbarrier / TMA helpers ------------------------------------------------
__device__ __forceinline__ unsigned smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for phase `parity` of `bar` to complete, for at most kWaitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}
__device__ __forceinline__ void tma_load_3d(float* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];\n" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}


// A CTA that timed out: record it, then let thread 0 wait (bounded) for the
// copies it issued and nobody consumed, so none lands after the CTA is gone.
template <int NST>
__device__ void give_up(uint64_t* full, int first_unconsumed, int issued) {
    if (threadIdx.x == 0) {
        atomicCAS(&g_dw_status, 0, (int)HC_ERR_TIMEOUT);
        for (int j = first_unconsumed; j < issued; j++)
            mbar_wait(full + (j % NST), (unsigned)((j / NST) & 1));
    }
}

// ---- the stencil ------------------------------------------------------------
// acc[r][jj] += sum_{u,v} wt[u][v] * tile[row0 + r + u][4*lane + jj + v - P + 4];
// done(r) runs as soon as output row r has all its terms (after input row r + K - 1),
// so a row's store issues while the later rows compute.
template <int K, typename Done>
__device__ __forceinline__ void stencil_8x4(const float* sm, int row0, int lane, const float (&wt)[K][K],
                                            float (&acc)[8][4], Done&& done) {
    constexpr int P = (K - 1) / 2;
#pragma unroll
    for (int i = 0; i < 8 + 2 * P; i++) {
        const float4* rp = reinterpret_cast<const float4*>(sm + (row0 + i) * SMW + 4 * lane);
        const float4 a = rp[0], b = rp[1], c = rp[2];
        const float xs[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int r = 0; r < 8; r++) {
            const int u = i - r;
            if (u >= 0 && u < K) {
#pragma unroll
                for (int jj = 0; jj < 4; jj++)
#pragma unroll
                    for (int v = 0; v < K; v++) acc[r][jj] = fmaf(wt[u][v], xs[jj + v - P + 4], acc[r][jj]);
            }
        }
        if (i >= K - 1) done(i - (K - 1));
    }
}

// Half-block forms used by the backward: rows row0 .. row0+3 of the block
// (done(r) as in stencil_8x4).
template <int K, typename Done>
__device__ __forceinline__ void stencil_4x4(const float* sm, int row0, int lane, const float (&wt)[K][K],
                                            float (&acc)[4][4], Done&& done) {
    constexpr int P = (K - 1) / 2;
#pragma unroll
    for (int i = 0; i < 4 + 2 * P; i++) {
        const float4* rp = reinterpret_cast<const float4*>(sm + (row0 + i) * SMW + 4 * lane);
        const float4 a = rp[0], b = rp[1], c = rp[2];
        const float xs[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const int u = i - r;
            if (u >= 0 && u < K) {
#pragma unroll
                for (int jj = 0; jj < 4; jj++)
#pragma unroll
                    for (int v = 0; v < K; v++) acc[r][jj] = fmaf(wt[u][v], xs[jj + v - P + 4], acc[r][jj]);
            }
        }
        if (i >= K - 1) done(i - (K - 1));
    }
}

template <int K>
__device__ __forceinline__ void correlate_4x4(const float* sm, int row0, int lane, const float (&g)[4][4],
                                              float (&gw)[K][K]) {
    constexpr int P = (K - 1) / 2;
#pragma unroll
    for (int i = 0; i < 4 + 2 * P; i++) {
        const float4* rp = reinterpret_cast<const float4*>(sm + (row0 + i) * SMW + 4 * lane);
        const float4 a = rp[0], b = rp[1], c = rp[2];
        const float xr[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const int u = i - r;
            if (u >= 0 && u < K) {
#pragma unroll
                for (int jj = 0; jj < 4; jj++)
#pragma unroll
                    for (int v = 0; v < K; v++) gw[u][v] = fmaf(g[r][jj], xr[jj + v - P + 4], gw[u][v]);
            }
        }
    }
}

struct Sched {
    int N, C, H, W, col_tiles, items;
    // item order.  1: (c, n, column tile), contiguous ranges per CTA.  0: (c, column
    // tile, n), contiguous ranges per CTA.  2: the column tiles in blocks of tb; CTA b
    // keeps tile b % tb of a block and walks (tile block, c, n), n fastest; the tb CTAs
    // of a group share one contiguous range of that sequence, so neighbouring tiles
    // read their common halo strips at about the same time (L2 hits) while each CTA's
    // runs of one (c, column tile) stay whole.  (tb divides col_tiles and the grid is
    // a multiple of tb.)
    int tile_fastest;
    int tb;
    // The column tiles the items cover: tile k (0 <= k < col_tiles) is column tile
    // ct_base + k * ct_step of the output (all of them: 0, 1; a rank's interior or
    // edge tiles: see the rank entry points).  xo: the column of the x (and
    // grad_output) tensor maps where the block's column 0 sits (4 in the
    // halo-padded layout, else 0).
    int ct_base, ct_step, xo;
    __device__ __forceinline__ int col(int k) const { return ct_base + k * ct_step; }
    __device__ __forceinline__ void decode(int item, int& n, int& c, int& ct) const {
        if (tile_fastest == 2) {
            n = item % N;
            const int rest = item / N;
            c = rest % C;
            ct = (rest / C) * tb + (int)blockIdx.x % tb;
        } else if (tile_fastest) {
            ct = item % col_tiles;
            const int rest = item / col_tiles;
            n = rest % N;
            c = rest / N;
        } else {
            n = item % N;
            const int rest = item / N;
            ct = rest % col_tiles;
            c = rest / col_tiles;
        }
    }
    // the item after (n, c, ct) in this order, without divisions
    __device__ __forceinline__ void next(int& n, int& c, int& ct) const {
        if (tile_fastest == 2) {
            if (++n == N) {
                n = 0;
                if (++c == C) {  // the next tile block
                    c = 0;
                    ct += tb;
                }
            }
        } else if (tile_fastest) {
            if (++ct == col_tiles) {
                ct = 0;
                if (++n == N) {
                    n = 0;
                    ++c;
                }
            }
        } else if (++n == N) {
            n = 0;
            if (++ct == col_tiles) {
                ct = 0;
                ++c;
            }
        }
    }
    // This CTA's jobs [j0, j1) when each item is split into `ntiles` row-tile jobs
    // and the split falls between any two jobs (item = job / ntiles).
    __device__ __forceinline__ void job_range(int ntiles, long long& j0, long long& j1) const {
        const bool grouped = tile_fastest == 2;
        const long long total = (grouped ? (long long)N * C * (col_tiles / tb) : (long long)items) * ntiles;
        const int idx = grouped ? (int)blockIdx.x / tb : (int)blockIdx.x;
        const int parts = grouped ? (int)gridDim.x / tb : (int)gridDim.x;
        j0 = idx * total / parts;
        j1 = (idx + 1) * total / parts;
    }
    __device__ __forceinline__ void range(int& i0, int& i1) const {
        if (tile_fastest == 2) {  // items here index (tile block, c, n) of the CTA's own tile in each block
            const int g = blockIdx.x / tb, groups = gridDim.x / tb;
            const long long per = (long long)N * C * (col_tiles / tb);
            i0 = (int)(g * per / groups);
            i1 = (int)((g + 1) * per / groups);
            return;
        }
        i0 = (int)((long long)blockIdx.x * items / gridDim.x);
        i1 = (int)((long long)(blockIdx.x + 1) * items / gridDim.x);
    }
};

// ---- forward ----------------------------------------------------------------
// Warps run through the CTA's jobs independently: a warp waits for its job's
// stage to fill, computes, and counts itself done with the stage; the last
// warp done refills the stage with the job NSTAGE ahead, so no job ends in a
// CTA-wide barrier.  A warp that changes channel reads the K*K weights straight
// from global memory (L1 / L2 hits after the first warp).
template <int K>
__global__ void __launch_bounds__(FWD_WARPS * 32, FWD_CTAS)
    dw_fwd_kernel(const __grid_constant__ CUtensorMap xmap, const float* __restrict__ w,
                  const float* __restrict__ bias, float* __restrict__ y, Sched sc) {
    using G = Geo<K, FWD_WARPS>;
    constexpr int P = G::P, TH = G::TH, KK = K * K;
    extern __shared__ __align__(1024) float smem[];
    float* tiles = smem;                                               // [NSTAGE][TILE]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + NSTAGE * G::TILE);
    int* done = reinterpret_cast<int*>(full + NSTAGE);                 // [NSTAGE] warps finished with the stage
    int* issued = done + NSTAGE;                                       // jobs whose copies have been issued
    int* failed = issued + 1;                                          // a warp gave up waiting
    const int tid = threadIdx.x, lane = tid & 31;
    int i0, i1;
    sc.range(i0, i1);
    if (i0 >= i1) return;
    const int ntiles = (sc.H + TH - 1) / TH;
    const int jobs = (i1 - i0) * ntiles;

    auto issue = [&](int q) {
        int n, c, ct;
        sc.decode(i0 + q / ntiles, n, c, ct);
        uint64_t* bar = full + (q % NSTAGE);
        mbar_expect_tx(bar, G::BYTES);
        tma_load_3d(tiles + (q % NSTAGE) * G::TILE, &xmap, sc.xo + sc.col(ct) * TW - 4, (q % ntiles) * TH - P,
                    n * sc.C + c, bar);
    };
    if (tid == 0) {
        for (int s = 0; s < NSTAGE; s++) {
            mbar_init(full + s, 1);
            done[s] = 0;
        }
        *failed = 0;
        fence_barrier_init();
        const int first = jobs < NSTAGE ? jobs : NSTAGE;
        for (int j = 0; j < first; j++) issue(j);
        *issued = first;
    }
    __syncthreads();

    const int warp = tid >> 5;
    float wt[K][K];
    float bv = 0.0f;
    int cur_c = -1;
    // this warp's job: item (n, c, ct) and row tile t, advanced one job at a time
    int n, c, ct, t = 0, s = 0;
    unsigned ph = 0;  // phase of stage s's barrier this job waits for
    sc.decode(i0, n, c, ct);
    for (int q = 0; q < jobs; q++) {
        if (c != cur_c) {
#pragma unroll
            for (int u = 0; u < K; u++)
#pragma unroll
                for (int v = 0; v < K; v++) wt[u][v] = __ldg(w + c * KK + u * K + v);
            bv = bias ? __ldg(bias + c) : 0.0f;
            cur_c = c;
        }
        const bool ok = __all_sync(0xffffffffu, mbar_wait(full + s, ph));
        if (!ok) {
            if (lane == 0) {
                atomicCAS(&g_dw_status, 0, (int)HC_ERR_TIMEOUT);
                *reinterpret_cast<volatile int*>(failed) = 1;
            }
            break;
        }
        const float* sm = tiles + s * G::TILE;
        float acc[8][4];
#pragma unroll
        for (int r = 0; r < 8; r++)
#pragma unroll
            for (int jj = 0; jj < 4; jj++) acc[r][jj] = bv;
        float* yp = y + ((long long)(n * sc.C + c) * sc.H) * sc.W + sc.col(ct) * TW + 4 * lane;
        stencil_8x4<K>(sm, warp * 8, lane, wt, acc, [&](int r) {
            const int h = t * TH + warp * 8 + r;
            if (h < sc.H)
                *reinterpret_cast<float4*>(yp + (long long)h * sc.W) =
                    make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        });
        __syncwarp();  // the warp's reads of the stage are done
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(done + s, 1) == FWD_WARPS - 1) {  // the last warp out refills the stage
                done[s] = 0;
                __threadfence_block();
                if (q + NSTAGE < jobs) {
                    issue(q + NSTAGE);
                    atomicAdd(issued, 1);
                }
            }
        }
        if (++s == NSTAGE) {
            s = 0;
            ph ^= 1u;
        }
        if (++t == ntiles) {
            t = 0;
            sc.next(n, c, ct);
        }
    }
    // A warp that gave up: wait (bounded) for the copies still in flight, so
    // none lands after the CTA is gone.  At most NSTAGE jobs are outstanding.
    __syncthreads();
    if (tid == 0 && *failed) {
        const int last = *issued;
        for (int j = last - NSTAGE > 0 ? last - NSTAGE : 0; j < last; j++)
            mbar_wait(full + (j % NSTAGE), (unsigned)((j / NSTAGE) & 1));
    }
}

// ---- backward ---------------------------------------------------------------
// Job cursor of the backward with row shards.  A CTA's jobs go run by run (a run:
// its items of one (c, column tile), n fastest), within a run row shard by row
// shard, within a row shard item by item and, per item, over the row shard's
// tpr row tiles; the weight gradient of one (run, row shard) is flushed at its
// last job.  Advanced one job at a time: one decode per run, no per-job division.
struct RowJobs {
    int item, seg, tt;  // this job: item, row shard, row tile within the row shard
    int rs, re;         // this run's items [rs, re)
    int n, c, ct;       // the item's coordinates
    int n_rs;           // the image of item rs
    __device__ __forceinline__ void start(const Sched& sc, int i0, int i1) {
        rs = i0;
        const int e = (i0 / sc.N + 1) * sc.N;
        re = e < i1 ? e : i1;
        item = rs;
        seg = tt = 0;
        sc.decode(rs, n, c, ct);
        n_rs = n;
    }
    __device__ __forceinline__ int t(int tpr) const { return seg * tpr + tt; }
    __device__ __forceinline__ bool seg_end(int tpr) const { return item == re - 1 && tt == tpr - 1; }
    __device__ __forceinline__ void advance(const Sched& sc, int Sh, int tpr, int i1) {
        if (++tt < tpr) return;
        tt = 0;
        if (++item < re) {  // the next image of the run (n fastest)
            ++n;
            return;
        }
        item = rs;
        n = n_rs;
        if (++seg < Sh) return;  // the run again, in the next row shard
        seg = 0;
        rs = re;  // the next run starts on a run boundary
        if (rs >= i1) return;  // past the CTA's last job
        re = rs + sc.N < i1 ? rs + sc.N : i1;
        item = rs;
        sc.decode(rs, n, c, ct);
        n_rs = n;
    }
};

struct BwdArgs {
    const float* w;
    float* gx;
    const float* gres;  // nullable: added to grad_input (a residual branch's gradient), same layout as gx
    float* tile_part;
    int tiles_per_shard;
    int want_wb;
    int S, Sh, hlo;  // column shards, row shards, rows per row shard (a multiple of TH when Sh > 1)
    int slots;       // partial slots per (grid shard, c, tile)
    int pieces;      // without row shards: a slot per piece of a run (else per job)
};

// ROWS: row shards present (a.Sh > 1); RES: a residual gradient is added to
// grad_input (a.gres).  Separate instantiations, so that the plain kernel
// carries none of their bookkeeping.
template <int K, bool ROWS, bool RES>
__global__ void __launch_bounds__(2 * BWD_WARPS * 32, BWD_CTAS)
    dw_bwd_kernel(const __grid_constant__ CUtensorMap gymap, const __grid_constant__ CUtensorMap xmap, BwdArgs a,
                  Sched sc) {
    using G = Geo<K, BWD_WARPS>;
    constexpr int P = G::P, TH = G::TH, KK = K * K;
    extern __shared__ __align__(1024) float smem[];
    float* tiles = smem;                                   // [BWD_NSTAGE][gy, x][TILE]
    float* red = smem + 2 * BWD_NSTAGE * G::TILE;          // [BWD_WARPS][KK + 1]
    uint64_t* full = reinterpret_cast<uint64_t*>(red + BWD_WARPS * WSLOT);
    RowJobs& rj = *reinterpret_cast<RowJobs*>(full + BWD_NSTAGE);  // the issuer's cursor (row shards)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = (sc.H + TH - 1) / TH;
    // Without row shards the CTA's jobs are a contiguous run of (item, row tile)
    // pairs that may start and end inside an item (t0: the first job's row tile);
    // with row shards whole items.
    int i0, i1, jobs, t0 = 0;
    if (ROWS) {
        sc.range(i0, i1);
        if (i0 >= i1) return;
        jobs = (i1 - i0) * ntiles;
    } else {
        long long j0, j1;
        sc.job_range(ntiles, j0, j1);
        if (j0 >= j1) return;
        jobs = (int)(j1 - j0);
        i0 = (int)(j0 / ntiles);
        t0 = (int)(j0 - (long long)i0 * ntiles);
        i1 = i0;  // unused without row shards
    }
    const bool want_wb = a.want_wb != 0;

    // Jobs: items run (c, column tile, n), n fastest; a run is this CTA's jobs of
    // one (c, column tile).  Without row shards the jobs go item by item, tile by
    // tile; with row shards as RowJobs walks them.
    const int tpr = ntiles / a.Sh;  // row tiles per row shard (row shards only)

    // The issuer thread issues the jobs in order; its cursor ((in_, ic, ict, it), or rj in
    // shared memory with row shards: no registers held by every thread) advances one job
    // at a time (no divisions).
    int in_ = 0, ic = 0, ict = 0, it = t0;
    if (!ROWS) sc.decode(i0, in_, ic, ict);
    auto issue = [&](int q) {
        (void)q;
        int n, c, ct, t;
        if (ROWS) {
            n = rj.n, c = rj.c, ct = rj.ct, t = rj.t(tpr);
            rj.advance(sc, a.Sh, tpr, i1);
        } else {
            n = in_, c = ic, ct = ict, t = it;
            if (++it == ntiles) {
                it = 0;
                sc.next(in_, ic, ict);
            }
        }
        uint64_t* bar = full + (q % BWD_NSTAGE);
        float* st = tiles + (q % BWD_NSTAGE) * 2 * G::TILE;
        mbar_expect_tx(bar, want_wb ? 2 * G::BYTES : G::BYTES);
        const int x0 = sc.xo + sc.col(ct) * TW - 4, y0 = t * TH - P, z = n * sc.C + c;
        tma_load_3d(st, &gymap, x0, y0, z, bar);
        if (want_wb) tma_load_3d(st + G::TILE, &xmap, x0, y0, z, bar);
    };
    // the copies are issued by lane 0 of the first weight-gradient warp: the
    // grad_input role is the longer one, so none of its warps waits on an issue
    const int issuer = BWD_WARPS * 32;
    if (tid == issuer) {
        for (int s = 0; s < BWD_NSTAGE; s++) mbar_init(full + s, 1);
        if (ROWS) rj.start(sc, i0, i1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == issuer)
        for (int j = 0; j < BWD_NSTAGE && j < jobs; j++) issue(j);

    // The ring, shared by both roles: every warp waits for job q's stage, does
    // its role's work on it, and the stage is refilled after a CTA barrier.
    // work(s, n, c, ct, t, flush): s = the job's stage; flush = the last job of a
    // weight-gradient run (segment).  Returns false when a wait timed out.
    auto ring = [&](auto&& on_channel, auto&& work) {
        int cur_c = -1;
        // without row shards: job q's item (n, c, ct) and row tile t, advanced one job at a time
        int n, c, ct, t = t0, s = 0;
        unsigned ph = 0;  // phase of stage s's barrier this job waits for
        RowJobs cur{};
        if (!ROWS) sc.decode(i0, n, c, ct);
        else cur.start(sc, i0, i1);
        for (int q = 0; q < jobs; q++) {
            bool flush;
            if (ROWS) {
                n = cur.n, c = cur.c, ct = cur.ct, t = cur.t(tpr);
                flush = cur.seg_end(tpr);  // the last job of a (run, row shard) segment
            } else {
                // the last job of a run: the CTA's last job, or the last row tile of
                // image N - 1 (the next job is another (c, column tile))
                flush = q + 1 == jobs || (t == ntiles - 1 && n == sc.N - 1);
            }
            if (c != cur_c) {
                on_channel(c);
                cur_c = c;
            }
            // A wait that ran out is acted on at the job's end, where every warp meets
            // (one CTA barrier per job): all warps still run the job (the named barrier
            // of the weight-gradient flush needs every one of its warps; the stage's
            // contents are then not valid, and the call reports HC_ERR_TIMEOUT), then
            // the CTA gives up.
            const bool ok = mbar_wait(full + s, ph);
            work(s, n, c, ct, t, flush);
            if (__syncthreads_or(!ok)) {  // every warp is done with this stage
                give_up<BWD_NSTAGE>(full, q, q + BWD_NSTAGE < jobs ? q + BWD_NSTAGE : jobs);
                return;
            }
            if (tid == issuer && q + BWD_NSTAGE < jobs) issue(q + BWD_NSTAGE);
            if (++s == BWD_NSTAGE) {
                s = 0;
                ph ^= 1u;
            }
            if (ROWS) {
                cur.advance(sc, a.Sh, tpr, i1);
            } else if (++t == ntiles) {
                t = 0;
                sc.next(n, c, ct);
            }
        }
    };

    if (warp < BWD_WARPS) {
        // grad_input warps: the flipped stencil on grad_output, 8 rows each in two 4-row halves
        float wf[K][K];
        ring(
            [&](int c) {
#pragma unroll
                for (int u = 0; u < K; u++)
#pragma unroll
                    for (int v = 0; v < K; v++) wf[u][v] = __ldg(a.w + c * KK + (K - 1 - u) * K + (K - 1 - v));
            },
            [&](int s, int n, int c, int ct, int t, bool) {
                if (!a.gx) return;
                const float* gys = tiles + s * 2 * G::TILE;
                const long long off = ((long long)(n * sc.C + c) * sc.H) * sc.W + sc.col(ct) * TW + 4 * lane;
                float* gp = a.gx + off;
#pragma unroll 1
                for (int half = 0; half < 2; half++) {
                    const int row0 = warp * 8 + 4 * half;
                    // the residual rows, loaded before the stencil so their latency is hidden
                    float4 res[4];
#pragma unroll
                    for (int r = 0; r < 4; r++) {
                        const int h = t * TH + row0 + r;
                        res[r] = RES && h < sc.H ? __ldg(reinterpret_cast<const float4*>(a.gres + off + (long long)h * sc.W))
                                                 : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    }
                    float acc[4][4];
#pragma unroll
                    for (int r = 0; r < 4; r++)
#pragma unroll
                        for (int jj = 0; jj < 4; jj++) acc[r][jj] = 0.0f;
                    stencil_4x4<K>(gys, row0, lane, wf, acc, [&](int r) {
                        const int h = t * TH + row0 + r;
                        if (h < sc.H)
                            *reinterpret_cast<float4*>(gp + (long long)h * sc.W) =
                                RES ? make_float4(acc[r][0] + res[r].x, acc[r][1] + res[r].y, acc[r][2] + res[r].z,
                                                  acc[r][3] + res[r].w)
                                    : make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
                    });
                }
            });
    } else {
        // weight / bias gradient warps: the correlation of the same rows with x,
        // accumulated in registers over a run and flushed at its end
        const int wg = warp - BWD_WARPS, wtid = tid - BWD_WARPS * 32;
        float gw[K][K];
        float gbs = 0.0f;
#pragma unroll
        for (int u = 0; u < K; u++)
#pragma unroll
            for (int v = 0; v < K; v++) gw[u][v] = 0.0f;
        // Partial slots of one (grid shard, c, tile), a.slots of them: with row shards
        // one per image, a run's total in its first slot and zeros in the rest.
        // Without them either one per piece of a run (a.pieces: the run's jobs in one
        // CTA range; the piece's index is the number of range starts inside the run
        // before it, and the run's last piece zeroes the slots that no piece takes)
        // or one per (image, row tile) as with row shards.  Every slot is written once.
        const int slots = a.slots;
        // Only the CTA's first run can start before its range (sc.job_range: every
        // range holds a job when a.pieces is set): its piece is the CTA's range index
        // less that of the range holding the run's first job; every later run starts
        // in this CTA, at piece 0.
        int next_piece = 0;
        if (!ROWS && a.pieces) {
            const bool grouped = sc.tile_fastest == 2;
            const long long L = (long long)sc.N * ntiles;
            const long long T = (grouped ? (long long)sc.N * sc.C * (sc.col_tiles / sc.tb) : (long long)sc.items) * ntiles;
            const long long parts = grouped ? gridDim.x / sc.tb : gridDim.x;
            const long long g = grouped ? blockIdx.x / sc.tb : blockIdx.x;
            const long long run0 = (g * T / parts) / L;  // the run of the CTA's first job
            // the last range index h with h * T / parts <= run0 * L
            const long long gfirst = ((run0 * L + 1) * parts + T - 1) / T - 1;
            next_piece = (int)(g - gfirst);
        }
        int run_m0 = -1;  // first slot of the current run (piece)
        ring([](int) {},
             [&](int s, int n, int c, int ct, int t, bool flush) {
                 if (RES && !ROWS && a.gx) {
                     // the next job's residual rows into L2 for the grad_input warp of the same
                     // rows (the longer role): one 128-byte line per lane, row lane / 4 of the
                     // warp's eight, quarter lane % 4 of the 512-byte segment, so that warp's
                     // residual loads are L2 hits rather than DRAM misses
                     int n2 = n, c2 = c, ct2 = ct, t2 = t + 1;
                     if (t2 == ntiles) {
                         t2 = 0;
                         sc.next(n2, c2, ct2);
                     }
                     const int h2 = t2 * TH + wg * 8 + (lane >> 2);
                     if (c2 < sc.C && ct2 < sc.col_tiles && h2 < sc.H) {  // not past the CTA's last item
                         const float* pf = a.gres + ((long long)(n2 * sc.C + c2) * sc.H + h2) * sc.W +
                                           sc.col(ct2) * TW + (lane & 3) * 32;
                         asm volatile("prefetch.global.L2 [%0];\n" ::"l"(pf));
                     }
                 }
                 if (!want_wb) return;
                 const int m = ROWS ? n : n * ntiles + t;
                 if (run_m0 < 0) {
                     run_m0 = !ROWS && a.pieces ? next_piece : m;
                     next_piece = 0;
                 }
                 const float* gys = tiles + s * 2 * G::TILE;
                 const float* xs = gys + G::TILE;
#pragma unroll 1
                 for (int half = 0; half < 2; half++) {
                     const int row0 = wg * 8 + 4 * half;
                     float g[4][4];
#pragma unroll
                     for (int r = 0; r < 4; r++) {
                         const float4 v4 = *reinterpret_cast<const float4*>(gys + (P + row0 + r) * SMW + 4 + 4 * lane);
                         g[r][0] = v4.x;
                         g[r][1] = v4.y;
                         g[r][2] = v4.z;
                         g[r][3] = v4.w;
                         gbs += (v4.x + v4.y) + (v4.z + v4.w);
                     }
                     correlate_4x4<K>(xs, row0, lane, g, gw);
                 }
                 // flush at the end of a (c, column tile) run; with row shards, at the end
                 // of each row-shard segment of the run (its partial belongs to that grid shard)
                 if (!flush) return;
#pragma unroll
                 for (int u = 0; u < K; u++)
#pragma unroll
                     for (int v = 0; v < K; v++) {
                         float sum = gw[u][v];
#pragma unroll
                         for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                         if (lane == 0) red[wg * WSLOT + u * K + v] = sum;
                         gw[u][v] = 0.0f;
                     }
                 float sum = gbs;
#pragma unroll
                 for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                 if (lane == 0) red[wg * WSLOT + KK] = sum;
                 gbs = 0.0f;
                 asm volatile("bar.sync 1, %0;\n" ::"n"(BWD_WARPS * 32) : "memory");  // the weight-gradient warps
                 if (wtid <= KK) {
                     float tot = 0.0f;
#pragma unroll
                     for (int k = 0; k < BWD_WARPS; k++) tot += red[k * WSLOT + wtid];
                     const int r = sc.col(ct) / a.tiles_per_shard, tt = sc.col(ct) - r * a.tiles_per_shard;
                     const int qs = ROWS ? (t * TH) / a.hlo * a.S + r : r;  // grid shard
                     float* slot = a.tile_part + (((long long)qs * sc.C + c) * a.tiles_per_shard + tt) * slots * (KK + 1);
                     if (!ROWS && a.pieces) {
                         slot[(long long)run_m0 * (KK + 1) + wtid] = tot;
                         if (t == ntiles - 1 && n == sc.N - 1)  // the run's last piece
                             for (int k = run_m0 + 1; k < slots; k++) slot[(long long)k * (KK + 1) + wtid] = 0.0f;
                     } else {
                         for (int k = run_m0; k <= m; k++) slot[(long long)k * (KK + 1) + wtid] = k == run_m0 ? tot : 0.0f;
                     }
                 }
                 run_m0 = -1;
             });
    }
}

// Shard partials: gwp[r][c][k] = sum over shard r's slots of the partials (tile
// tt, then the tile's slots, ascending); gbp[r][c] likewise from the last entry.  One thread per
// (c, k) walks the shards in order and also writes the full gradients
// gw[c][k] / gb[c] (either may be null): the shard partials added from shard 0
// up, the order hc_conv2d_bwd's shard sum uses.
__global__ void dw_shard_partials_kernel(const float* __restrict__ tile_part, float* __restrict__ gwp,
                                         float* __restrict__ gbp, float* __restrict__ gw, float* __restrict__ gb,
                                         int Q, int C, int rows, int KK) {
    constexpr int B = 16;  // loads in flight per thread
    const long long total = (long long)C * (KK + 1);
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        const int k = (int)(q % (KK + 1));
        const int c = (int)(q / (KK + 1));
        // the (shard r, slot m) pairs in order, r slowest: loaded B at a time, added one
        // by one (slots ascending within a shard, shards ascending into the total)
        const long long all = (long long)Q * rows;
        float s = 0.0f, tot = 0.0f;
        int lr = 0, lm = 0, ar = 0, am = 0;  // load and add cursors (shard, slot)
        for (long long i0 = 0; i0 < all; i0 += B) {
            float v[B];
#pragma unroll
            for (int i = 0; i < B; i++) {
                v[i] = 0.0f;
                if (i0 + i < all) {
                    v[i] = __ldg(tile_part + (((long long)lr * C + c) * rows + lm) * (KK + 1) + k);
                    if (++lm == rows) {
                        lm = 0;
                        ++lr;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < B; i++) {
                if (i0 + i >= all) break;
                s += v[i];
                if (++am == rows) {  // shard ar complete
                    const long long rc = (long long)ar * C + c;
                    if (k < KK) {
                        if (gwp) gwp[rc * KK + k] = s;
                    } else if (gbp) {
                        gbp[rc] = s;
                    }
                    tot += s;
                    s = 0.0f;
                    am = 0;
                    ++ar;
                }
            }
        }
        if (k < KK) {
            if (gw) gw[(long long)c * KK + k] = tot;
        } else if (gb) {
            gb[c] = tot;
        }
    }
}


// The same sums with one lane per shard: lanes r = 0..Q-1 of one (c, k) group
// (Q divides 32, so a group never straddles a warp) each add their shard's
// slots in order and write gwp / gbp, then the group's lane 0 gathers the Q
// shard sums by shuffles and adds them from shard 0 up -- the order of
// dw_shard_partials_kernel, with Q times the threads in flight.
__global__ void dw_shard_partials_lanes_kernel(const float* __restrict__ tile_part, float* __restrict__ gwp,
                                               float* __restrict__ gbp, float* __restrict__ gw,
                                               float* __restrict__ gb, int Q, int C, int rows, int KK) {
    constexpr int B = 16;  // loads in flight per thread
    const long long total = (long long)C * (KK + 1) * Q;
    const int lane = threadIdx.x & 31;
    // every lane of a warp runs the same number of iterations (total is a multiple of Q,
    // and of the whole grid's stride only by chance), so the shuffles see the whole group
    for (long long base = (long long)blockIdx.x * blockDim.x; base < total; base += (long long)gridDim.x * blockDim.x) {
        const long long t = base + threadIdx.x;
        const bool live = t < total;
        const int r = (int)(t % Q);
        const long long ck = t / Q;
        const int k = (int)(ck % (KK + 1));
        const int c = (int)(ck / (KK + 1));
        float s = 0.0f;
        if (live) {
            const float* src = tile_part + ((long long)r * C + c) * rows * (KK + 1) + k;
            for (int m0 = 0; m0 < rows; m0 += B) {
                float v[B];
#pragma unroll
                for (int i = 0; i < B; i++) v[i] = m0 + i < rows ? __ldg(src + (long long)(m0 + i) * (KK + 1)) : 0.0f;
#pragma unroll
                for (int i = 0; i < B; i++)
                    if (m0 + i < rows) s += v[i];
            }
            const long long rc = (long long)r * C + c;
            if (k < KK) {
                if (gwp) gwp[rc * KK + k] = s;
            } else if (gbp) {
                gbp[rc] = s;
            }
        }
        // the group's lane 0 adds the shard sums in order
        float tot = s;
        const int g0 = lane - r;  // this group's first lane
        for (int j = 1; j < Q; j++) {
            const float o = __shfl_sync(0xffffffffu, s, g0 + j);
            if (r == 0) tot += o;
        }
        if (live && r == 0) {
            if (k < KK) {
                if (gw) gw[(long long)c * KK + k] = tot;
            } else if (gb) {
                gb[c] = tot;
            }
        }
    }
}

// Tensor map of an NCHW fp32 tensor viewed as [N*C][H][pitch] (pitch 0: W),
// box = one staged tile.
template <int K, int WARPS>
hc_status plane_map(CUtensorMap* m, const float* base, const hc_conv_desc* d, int pitch) {
    const uint64_t wp = pitch > 0 ? (uint64_t)pitch : (uint64_t)d->W;
    const uint64_t dims[3] = {wp, (uint64_t)d->H, (uint64_t)d->N * d->C_in};
    const uint64_t strides[2] = {wp * 4, (uint64_t)d->H * wp * 4};
    const uint32_t box[3] = {(uint32_t)SMW, (uint32_t)Geo<K, WARPS>::R, 1};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Weight-gradient partial slots per (grid shard, channel, column tile) of the
// backward, at most: one per image with row shards, else one per (image, row
// tile) (a launch over every tile uses one per piece of a run, no more).
long long bwd_slots(const hc_conv_desc* d, const Plan& p) {
    constexpr int TH = Geo<3, BWD_WARPS>::TH;  // the same for every K
    return p.Sh > 1 ? (long long)d->N : (long long)d->N * ((d->H + TH - 1) / TH);
}

Sched sched_of(const hc_conv_desc* d, int* grid, int tile_fastest, int ctas_per_sm, const DwLayout& lay) {
    const int T = d->W / TW;
    Sched sc{d->N, d->C_in, d->H, d->W, T, 0, tile_fastest, 1, 0, 1, lay.xo};
    if (lay.tiles == HC_TILES_INTERIOR) {
        sc.ct_base = 1;
        sc.col_tiles = T > 2 ? T - 2 : 0;
    } else if (lay.tiles == HC_TILES_EDGE) {
        sc.ct_step = T > 1 ? T - 1 : 1;
        sc.col_tiles = T > 1 ? 2 : 1;
    }
    sc.items = d->N * d->C_in * sc.col_tiles;
    const int g = device_sm_count() * ctas_per_sm;
    *grid = g < sc.items ? g : sc.items;
    if (tile_fastest == 2) {
        // groups of tb CTAs: tb the largest divisor of col_tiles whose groups fill at
        // least 96 % of the CTAs (few block edges, whose halo strips miss L2), else the
        // divisor that fills the most; with none that fits, runs of one (c, column
        // tile) in contiguous ranges instead
        int best = 0, used = 0;
        for (int t = sc.col_tiles; t >= 1; t--) {
            if (sc.col_tiles % t) continue;
            const int u = (g / t) * t;
            if (u > 0 && (long long)u * 100 >= (long long)g * 96) {
                best = t;
                break;
            }
            if (u > used) {
                used = u;
                best = t;
            }
        }
        if (best > 0) {
            sc.tb = best;
            const long long per = (long long)d->N * d->C_in * (sc.col_tiles / best);
            const int groups = g / best;
            *grid = (int)((groups < per ? groups : per) * best);
        } else {
            sc.tile_fastest = 0;
        }
    }
    return sc;
}

template <int K>
hc_status fwd_k(const hc_conv_desc* d, const float* x, const float* w, const float* b, float* y, cudaStream_t st,
                const DwLayout& lay) {
    using G = Geo<K, FWD_WARPS>;
    CUtensorMap xm;
    hc_status s = plane_map<K, FWD_WARPS>(&xm, x, d, lay.pitch);
    if (s) return s;
    int grid;
    const Sched sc = sched_of(d, &grid, 1, FWD_CTAS, lay);  // horizontal neighbours back to back: their halos hit L2
    if (sc.items == 0) return HC_OK;
    const size_t smem = sizeof(float) * NSTAGE * G::TILE + NSTAGE * sizeof(uint64_t) + (NSTAGE + 2) * sizeof(int);
    static std::atomic<unsigned long long> attr{0};
    once_per_device(attr, [&] {
        return cudaFuncSetAttribute(dw_fwd_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
               cudaSuccess;
    });
    dw_fwd_kernel<K><<<grid, FWD_WARPS * 32, smem, st>>>(xm, w, b, y, sc);
    return launched("dw_fwd_kernel", st);
}

template <int K>
hc_status bwd_k(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* gy, float* gx,
                const float* gres, float* tile_part, float* gwp, float* gbp, float* gw, float* gb, bool want_wb,
                cudaStream_t st, const DwLayout& lay) {
    using G = Geo<K, BWD_WARPS>;
    if (!gx && !want_wb) return HC_OK;
    CUtensorMap gm, xm;
    hc_status s = plane_map<K, BWD_WARPS>(&gm, gy, d, lay.pitch);
    if (s || (s = plane_map<K, BWD_WARPS>(&xm, x, d, lay.pitch))) return s;
    int grid;
    // runs of one (c, column tile): gw stays in registers; column tiles side by side in CTA groups
    const Sched sc = sched_of(d, &grid, 2, BWD_CTAS, lay);
    const int tps = p.Wl / TW;
    const size_t smem = sizeof(float) * (2 * BWD_NSTAGE * G::TILE + BWD_WARPS * WSLOT) +
                        BWD_NSTAGE * sizeof(uint64_t) + sizeof(RowJobs);
    static std::atomic<unsigned long long> attr{0};
    once_per_device(attr, [&] {
        const auto A = cudaFuncAttributeMaxDynamicSharedMemorySize;
        return cudaFuncSetAttribute(dw_bwd_kernel<K, false, false>, A, (int)smem) == cudaSuccess &&
               cudaFuncSetAttribute(dw_bwd_kernel<K, true, false>, A, (int)smem) == cudaSuccess &&
               cudaFuncSetAttribute(dw_bwd_kernel<K, false, true>, A, (int)smem) == cudaSuccess &&
               cudaFuncSetAttribute(dw_bwd_kernel<K, true, true>, A, (int)smem) == cudaSuccess;
    });
    // partial slots per (grid shard, c, tile): a slot per piece of a run (the run's jobs in
    // one CTA range) when one launch covers every tile and every range holds a job, so
    // the shard-partials pass reads a few slots per run instead of one per job
    int slots = (int)bwd_slots(d, p), pieces = 0;
    if (p.Sh == 1 && lay.tiles == HC_TILES_ALL && sc.items) {
        const int ntiles = (d->H + G::TH - 1) / G::TH;
        const long long L = (long long)d->N * ntiles;
        const bool grouped = sc.tile_fastest == 2;
        const long long T = (grouped ? (long long)sc.N * sc.C * (sc.col_tiles / sc.tb) : (long long)sc.items) * ntiles;
        const long long m = T / (grouped ? grid / sc.tb : grid);  // jobs of the shortest range
        if (m >= 1) {
            pieces = 1;
            const long long most = (L - 1 + m - 1) / m + 1;  // ranges meeting L consecutive jobs
            slots = (int)(most < L ? most : L);
        }
    }
    BwdArgs a{w, gx, gx ? gres : nullptr, tile_part, tps, want_wb ? 1 : 0, p.S, p.Sh, p.Hlo, slots, pieces};
    const dim3 grd(grid), blk(2 * BWD_WARPS * 32);
    if (sc.items == 0) {
        s = HC_OK;
    } else if (a.gres) {
        if (p.Sh > 1)
            dw_bwd_kernel<K, true, true><<<grd, blk, smem, st>>>(gm, xm, a, sc);
        else
            dw_bwd_kernel<K, false, true><<<grd, blk, smem, st>>>(gm, xm, a, sc);
    } else if (p.Sh > 1) {
        dw_bwd_kernel<K, true, false><<<grd, blk, smem, st>>>(gm, xm, a, sc);
    } else {
        dw_bwd_kernel<K, false, false><<<grd, blk, smem, st>>>(gm, xm, a, sc);
    }
    if (sc.items) s = launched("dw_bwd_kernel", st);
    if (s || !want_wb || !lay.partials) return s;
    return launch_shard_partials(tile_part, gwp, gbp, gw, gb, p.Q, d->C_in, tps * slots, K * K, st);
}

}  // namespace

hc_status launch_shard_partials(const float* tile_part, float* gwp, float* gbp, float* gw, float* gb, int Q, int C,
                                int rows, int KK, cudaStream_t st) {
    if (Q > 1 && 32 % Q == 0) {  // one lane per shard
        const long long total = (long long)C * (KK + 1) * Q;
        long long blocks = (total + 127) / 128;
        if (blocks > 152LL * 16) blocks = 152LL * 16;
        dw_shard_partials_lanes_kernel<<<(unsigned)blocks, 128, 0, st>>>(tile_part, gwp, gbp, gw, gb, Q, C, rows, KK);
        return launched("dw_shard_partials_kernel", st);
    }
    const long long total = (long long)C * (KK + 1);
    // small blocks: the few thousand threads spread over all the SMs
    dw_shard_partials_kernel<<<(unsigned)((total + 63) / 64), 64, 0, st>>>(tile_part, gwp, gbp, gw, gb, Q, C, rows,
                                                                           KK);
    return launched("dw_shard_partials_kernel", st);
}

bool depthwise_supported(const hc_conv_desc* d, const Plan& p) {
    const int K = d->kh;
    // row shards: the backward splits its weight-gradient runs at row-shard ends,
    // which must fall on its row-tile boundaries (the forward computes the global
    // conv whatever the row shards)
    return d->groups == d->C_in && d->C_out == d->C_in && d->kh == d->kw && (K == 3 || K == 5 || K == 7) &&
           d->stride == 1 && d->padding == (K - 1) / 2 && p.Wl % TW == 0 &&
           (p.Sh == 1 || p.Hlo % Geo<3, BWD_WARPS>::TH == 0) &&
           (long long)d->N * d->C_in * (d->W / TW) < (1LL << 31);
}

size_t depthwise_bwd_ws_floats(const hc_conv_desc* d, const Plan& p) {
    const int K = d->kh;
    return (size_t)p.Q * d->C_in * (p.Wl / TW) * bwd_slots(d, p) * (K * K + 1);
}

hc_status launch_depthwise_fwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w,
                               const float* b, float* y, cudaStream_t st, const DwLayout& lay) {
    (void)p;
    switch (d->kh) {
        case 3: return fwd_k<3>(d, x, w, b, y, st, lay);
        case 5: return fwd_k<5>(d, x, w, b, y, st, lay);
        case 7: return fwd_k<7>(d, x, w, b, y, st, lay);
    }
    return HC_ERR_UNSUPPORTED;
}

hc_status launch_depthwise_bwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w,
                               const float* gy, float* gx, float* tile_part, float* gwp, float* gbp,
                               bool want_weight_grads, cudaStream_t st, const float* gres, float* gw, float* gb,
                               const DwLayout& lay) {
    switch (d->kh) {
        case 3: return bwd_k<3>(d, p, x, w, gy, gx, gres, tile_part, gwp, gbp, gw, gb, want_weight_grads, st, lay);
        case 5: return bwd_k<5>(d, p, x, w, gy, gx, gres, tile_part, gwp, gbp, gw, gb, want_weight_grads, st, lay);
        case 7: return bwd_k<7>(d, p, x, w, gy, gx, gres, tile_part, gwp, gbp, gw, gb, want_weight_grads, st, lay);
    }
    return HC_ERR_UNSUPPORTED;
}

hc_status dw_take_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_dw_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return HC_ERR_CUDA;
    }
    if (v) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_dw_status, &zero, sizeof(int));
    }
    return (hc_status)v;
}

}  // namespace hc
