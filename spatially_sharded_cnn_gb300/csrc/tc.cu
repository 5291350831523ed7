// tc.cu -- dense (groups = 1) convolution as an implicit GEMM on the 5th-
// generation tensor cores (tcgen05, accumulators in tensor memory), with
// FP32 accuracy from 3xTF32: every operand is split as a = a_hi + a_lo with
// a_hi = tf32(a), a_lo = tf32(a - a_hi), and each product is taken as
// a_hi*b_hi + a_hi*b_lo + a_lo*b_hi (the a_lo*b_lo term is below fp32
// rounding), all accumulated in fp32 in TMEM.
//
// The W shards (NVIDIA blog "Perception model training for autonomous
// vehicles with tensor parallelism", design section and Figures 1-2; kwkr.cn
// news/18980 section 2.2): an output tile is one row segment of a shard's
// owned output columns, so the TMA boxes that feed it read the halo columns
// from the neighbouring shards' blocks and zeros past the image edge (the
// copy engine's out-of-bounds fill); the weight gradient is accumulated per
// shard over that shard's own output columns (its _Partial value), split
// further along the pixels to fill the GPU, and summed in a fixed order.
//
// Passes (all share one persistent, warp-specialised kernel):
//   conv   (forward, and grad_input of a stride-1 conv as the conv of
//          grad_output with the flipped, transposed kernel):
//          D[m][px] = sum over taps (u,v) and BK-channel chunks of
//          A[m][(u,v,c)] * X[n][h+u-p][w+v-p][c]; A = weights, B = the
//          activation in NHWC (channels contiguous), one 4-D TMA box per
//          (tap, chunk).
//   wgrad  G[co][ci] of one tap = sum over a shard's pixels of
//          gy[co][px] * x[ci][px + tap], on bf16 pieces (below): A =
//          grad_output's pieces (pixels contiguous, K-major), B = x's pieces
//          in a channel-blocked NHWC copy read as MN-major tiles, so a tap's
//          row and column shift are box coordinates on dimensions that are
//          not the innermost one (which must start on a 16-byte boundary),
//          with zero fill past the image.  A unit covers two (tap,
//          128-channel) slots side by side, each its own box and its own
//          N = 128 MMAs (256 accumulator columns).  (A space-to-depth conv
//          on this path keeps a tf32 weight gradient over planar copies.)
// The tf32 operands are K-major tiles with the 128-byte swizzle (32 tf32 per
// row): kind::tf32 takes no MN-major operands on this part.
//
// 1x1 convolutions (stride 1, no padding), k = stride convs and the weight
// gradient of K x K convs take a second operand format: every
// value is split into three bf16 pieces, a = a0 + a1 + a2 with a0 = bf16(a),
// a1 = bf16(a - a0), a2 = bf16(a - a0 - a1) (both differences are exact in
// fp32), and each product is taken as the six terms a_i*b_j with i + j <= 2
// (the dropped terms are below 2^-24 of |a*b|).  Six bf16 MMAs cost the tensor
// time of three tf32 ones, and 16-bit operands may be MN-major, so the pieces
// of the 1x1 and space-to-depth convs keep the NCHW order of the tensors they
// come from: their conv passes read pixels as MN-major B tiles, their weight
// gradient reads them as K-major tiles, and no pass needs a transposed copy.
// The K x K weight gradient reads x's pieces from one NHWC copy (above).
//
// Accuracy: the tensor core's fp32 accumulation loses about one unit in the
// last place per MMA step, so a long K would lose ~1e-5.  The MMA warp
// therefore accumulates groups of 256 k-values (96 MMAs) in one of two TMEM
// buffers and the epilogue warps add the groups up in fp32 registers.
//
// Warp roles (320 threads, one CTA per SM): warp 0 issues TMA loads into an
// mbarrier-guarded shared-memory ring, warp 1 issues tcgen05.mma into the two
// TMEM buffers in turn, warps 2-9 (two per TMEM lane quarter, one column half
// each) drain finished groups (tcgen05.ld) and store the tile.  Every wait is
// bounded: on timeout the CTA records HC_ERR_TIMEOUT, drains its outstanding
// copies and MMAs, frees its tensor memory and exits.
#include "common.cuh"

namespace hc {
namespace {

constexpr int BM = 128;             // accumulator rows (TMEM lanes)
constexpr int BK = 32;              // tf32 per k-chunk = one 128-byte swizzle row
constexpr int ROWB = BK * 4;        // bytes per tile row
constexpr uint32_t SW_ATOM = 8 * ROWB;  // 8-row swizzle atom = stride between 8-row groups
constexpr int TC_SMEM_RING = 192 * 1024;
constexpr int TC_STAGE_OUT = 4096;  // per epilogue warp: a 32 x 32 fp32 output box, 128-byte swizzle
// weight-gradient tiles: 128 output channels x two slots of 128 input channels
// (a slot is one tap x one 128-channel block)
constexpr int WG_BN = 256;
constexpr int WG_SLOT = 128;
constexpr uint32_t WG_SLOT_BYTES = WG_SLOT * 128;  // one slot's hi (or lo) tile: 128 rows x 32 tf32
constexpr int BKH = 32;             // bf16 pieces: k-values per chunk (channels in conv mode, pixels in wgrad mode)
constexpr int TC_SMEM_MAX = TC_SMEM_RING + 1024 + 8 * TC_STAGE_OUT;  // dynamic shared memory of every launch at most
constexpr long long kWait = 4000000000LL;  // clock cycles, about 2 s

__device__ int g_tc_status;

// ---------------------------------------------------------------------------
// PTX wrappers
__device__ __forceinline__ unsigned su32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, unsigned n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, unsigned parity) {
    unsigned ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok)
                 : "r"(su32(b)), "r"(parity)
                 : "memory");
    return ok != 0;
}
// Bounded wait; also gives up early once another role has aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, unsigned parity, volatile int* abort_flag) {
    if (mbar_try(b, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try(b, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWait) {
            *abort_flag = 1;
            atomicCAS(&g_tc_status, 0, (int)HC_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}
__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* m, int c0, int c1, int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n" ::
            "r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(su32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_5d(void* dst, const CUtensorMap* m, int c0, int c1, int c2, int c3, int c4,
                                       uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, "
        "%6}], [%7];\n" ::"r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(su32(bar))
        : "memory");
}
// TMA store of a shared-memory box to global memory (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];\n" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(su32(src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// the shared-memory source of every committed store has been read
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
// generic-proxy shared-memory writes become visible to the async (TMA) proxy
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ void tc_alloc(uint32_t* slot, unsigned cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(su32(slot)), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, unsigned cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(su32(bar))
                 : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc], kind::tf32, one CTA.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 with bf16 A and B, one CTA.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// 32 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 format: start,
// leading and stride byte offsets in 16-byte units, version 1 at bit 46,
// layout type 2 = SWIZZLE_128B at bits 61-63).
// Other layout types: 4 = SWIZZLE_64B.  K-major swizzled tiles: LBO unused,
// SBO = the stride of 8-row groups; MN-major tiles: LBO = the stride of the
// 64-element (128-byte) MN blocks, SBO = the stride of 8-row K groups.
__device__ __forceinline__ uint64_t sdesc(const void* p, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                          uint32_t layout = 2) {
    uint64_t d = 0;
    d |= (uint64_t)((su32(p) >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)layout << 61;
    return d;
}
// Instruction descriptor, kind::tf32: D fp32, A and B tf32, majors, N, M.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, int a_mn_major, int b_mn_major) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)a_mn_major << 15) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, majors, N, M.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn_major, int b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn_major << 15) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
struct TcParams {
    int mode;       // 0: conv (forward / stride-1 grad_input), 1: weight gradient
    int units;      // work units
    int stages;     // ring depth
    int chunks;     // k-chunks per unit (conv mode)
    int group;      // k-chunks accumulated in TMEM before the epilogue adds them up in fp32
    int tma_store;  // conv mode without depth-to-space: store through ymap (TMA boxes)
    int fmt;        // operands: 0 tf32 [hi][lo] pairs, 1 three bf16 pieces (1x1 convolutions)
    int stage_bytes, a_piece, b_piece;  // bf16 pieces: ring stage, one piece of the A / B tile
    // conv mode
    int N, Ho, Wo, M, Kc, kh, kw, pad, tiles_w, mblocks;
    const float* bias;
    float* out;     // NCHW [N][M][Ho][Wo], or with d2s > 0 the image [N][d2s_c][Ho*d2s][Wo*d2s]
    int d2s, d2s_c; // depth-to-space store: row m = (u*d2s_c + c)*d2s + v goes to pixel (ho*d2s+u, wo*d2s+v)
    // wgrad mode
    int Co, Ci, S, J, own_w, nblocks, taps, row_chunks;  // S: grid shards Sh*Sw; row_chunks = own_w / BK
    int Sw, own_h;  // column shards; owned output rows per row shard (shard q = a*Sw + b)
    int slots;      // taps * nblocks: (tap, 128-channel block) pairs; a unit covers two slots
    int kvalid;     // bf16 weight gradient: input channels that exist (the slots' columns past them
                    // are not computed: the reduction never reads them)
    int bmn;        // bf16 weight gradient of a K x K conv: B MN-major from x's pieces in the
                    // channel-blocked NHWC layout, each slot its own box at the tap's (row, column)
                    // shift and its own N = 128 MMAs
    long long shard_chunks;                               // N * own_h * row_chunks
    float* part;    // [S][J][taps][Co][Ci]
};

struct Unit {
    int m0;             // first accumulator row (output channel)
    int n, ho, w0;      // conv: output row segment
    int tap, ci0, r, j; // wgrad
    long long c_begin, c_end;
};

__device__ __forceinline__ Unit decode(const TcParams& p, int t, int BN) {
    Unit u{};
    if (p.mode == 0) {
        u.m0 = (t % p.mblocks) * BM;
        int rest = t / p.mblocks;
        u.w0 = (rest % p.tiles_w) * BN;
        rest /= p.tiles_w;
        u.ho = rest % p.Ho;
        u.n = rest / p.Ho;
        u.c_begin = 0;
        u.c_end = p.chunks;
    } else {
        u.m0 = (t % p.mblocks) * BM;
        int rest = t / p.mblocks;
        const int pairs = (p.slots + 1) / 2;
        u.tap = rest % pairs;  // slot pair: slots 2*tap and 2*tap + 1
        rest /= pairs;
        u.j = rest % p.J;
        u.r = rest / p.J;
        u.c_begin = p.shard_chunks * u.j / p.J;
        u.c_end = p.shard_chunks * (u.j + 1) / p.J;
    }
    return u;
}

struct Smem {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t buf_full[2];
    uint64_t buf_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

constexpr int TC_EPI_WARPS = 8;                    // two per TMEM lane quarter, one column half each
constexpr int TC_THREADS = 32 * (2 + TC_EPI_WARPS);

// One persistent CTA per SM.  BN = accumulator columns (pixels of an output
// row segment in conv mode, input channels in wgrad mode).
// FMT: operand format (p.fmt), a template parameter so that each format's
// instantiation carries only its own producer and MMA code.
template <int BN, int FMT>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_conv_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                   const __grid_constant__ CUtensorMap ymap, TcParams p) {
    extern __shared__ __align__(1024) unsigned char dsmem[];
    unsigned char* ring = (unsigned char*)(((uintptr_t)dsmem + 1023) & ~(uintptr_t)1023);  // 128-byte swizzle atoms need 1 KB
    // TC_EPI_WARPS output boxes, 1 KB aligned, after a conv-mode ring of at most TC_SMEM_RING
    // bytes (a weight-gradient ring, which stores no boxes, may extend over them)
    unsigned char* stage_out = ring + TC_SMEM_RING;
    __shared__ Smem sh;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr uint32_t a_bytes = BM * ROWB;           // 128 rows x BK tf32
    constexpr uint32_t b_bytes = BN * ROWB;
    constexpr uint32_t stage_bytes = 2 * a_bytes + 2 * b_bytes;
    volatile int* abort_flag = &sh.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; s++) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&sh.buf_full[b], 1);
            mbar_init(&sh.buf_empty[b], TC_EPI_WARPS);
        }
        mbar_init(&sh.drain, 1);
        sh.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) tc_alloc(&sh.tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        long long it = 0;  // chunk counter = ring position
        for (int t = blockIdx.x; t < p.units && !*abort_flag; t += gridDim.x) {
            const Unit u = decode(p, t, BN);
            for (long long c = u.c_begin; c < u.c_end; c++, it++) {
                const int s = (int)(it % p.stages);
                if (it >= p.stages && !mbar_wait(&sh.empty[s], (unsigned)(((it / p.stages) - 1) & 1), abort_flag))
                    break;
                if (FMT == 1) {
                    // bf16 pieces: one box brings all three pieces of a tile
                    unsigned char* st = ring + (size_t)s * p.stage_bytes;
                    unsigned char* bdst = st + 3 * p.a_piece;
                    if (p.bmn) {
                        // K x K weight gradient: chunk c of shard r = (n, 32-pixel piece, ho),
                        // rows fastest, so the kernel rows of one column strip reuse its rows
                        // while they are in L2.  A = grad_output [3][N][Co][H][W], 128 channels
                        // x 32 pixels (K-major).  B, per slot: x [N][H][W][C/128][3][128], the
                        // slot's 128 channels (all three pieces) at 32 pixels of row ho + u - pad
                        // from column w + v - pad (MN-major; W is not the innermost dimension, so
                        // any shift is a plain coordinate; rows and columns past the image read
                        // zeros)
                        const int qa = u.r / p.Sw, qb = u.r - qa * p.Sw;
                        const int ho = qa * p.own_h + (int)(c % p.own_h);
                        const long long rest = c / p.own_h;
                        const int wc = (int)(rest % p.row_chunks), n = (int)(rest / p.row_chunks);
                        const int w = qb * p.own_w + wc * BKH;
                        const int slot_bytes = 3 * (p.b_piece / 2);
                        const int nsl = 2 * u.tap + 1 < p.slots ? 2 : 1;
                        mbar_expect_tx(&sh.full[s], (unsigned)(3 * p.a_piece + nsl * slot_bytes));
                        tma_5d(st, &amap, w, ho, u.m0, n, 0, &sh.full[s]);
                        for (int h = 0; h < nsl; h++) {
                            const int slot = 2 * u.tap + h;
                            const int tap = slot / p.nblocks, cb = slot - tap * p.nblocks;
                            const int uu = tap / p.kw, vv = tap - uu * p.kw;
                            tma_5d(bdst + h * slot_bytes, &bmap, 0, w + vv - p.pad, 6 * cb, ho + uu - p.pad, n,
                                   &sh.full[s]);
                        }
                        continue;
                    }
                    mbar_expect_tx(&sh.full[s], (unsigned)p.stage_bytes);
                    if (p.mode == 0) {
                        // A: weights [3][M][K], 128 rows x 32 k; B: activation [3][N][K][Ho*Wo],
                        // BN pixels x 32 channels (the tile starts on a 64-pixel block)
                        tma_3d(st, &amap, (int)c * BKH, u.m0, 0, &sh.full[s]);
                        tma_5d(bdst, &bmap, 0, (int)c * BKH, (u.ho * p.Wo + u.w0) / 64, u.n, 0, &sh.full[s]);
                    } else {
                        // pixel chunk c of shard r, along the row: (n, ho, 32-pixel piece), the
                        // piece fastest, so a box row (64 bytes) and its neighbour in the same
                        // 128-byte line are read one after the other (a 1x1 kernel has no taps
                        // that would reuse rows).  A = grad_output [3][N][Co][H][W], 128
                        // channels x 32 pixels; B = x, the 256 channels of the slot pair (past
                        // C_in the box reads zeros)
                        const int qa = u.r / p.Sw, qb = u.r - qa * p.Sw;
                        const int wc = (int)(c % p.row_chunks);
                        const long long rest = c / p.row_chunks;
                        const int ho = qa * p.own_h + (int)(rest % p.own_h), n = (int)(rest / p.own_h);
                        const int w = qb * p.own_w + wc * BKH;
                        tma_5d(st, &amap, w, ho, u.m0, n, 0, &sh.full[s]);
                        tma_5d(bdst, &bmap, w, ho, 2 * u.tap * WG_SLOT, n, 0, &sh.full[s]);
                    }
                    continue;
                }
                unsigned char* st = ring + (size_t)s * stage_bytes;
                const bool second = p.mode == 0 || 2 * u.tap + 1 < p.slots;  // wgrad: last pair may be half
                mbar_expect_tx(&sh.full[s], second ? stage_bytes : stage_bytes - b_bytes);
                if (p.mode == 0) {
                    const int cpt = p.Kc / BK;
                    const int tap = (int)(c / cpt), cb = (int)(c % cpt);
                    const int uu = tap / p.kw, vv = tap % p.kw;
                    const int ka = tap * p.Kc + cb * BK;
                    tma_3d(st, &amap, ka, u.m0, 0, &sh.full[s]);  // [hi][lo] x 128 rows
                    const int wx = u.w0 + vv - p.pad, hy = u.ho + uu - p.pad;
                    tma_5d(st + 2 * a_bytes, &bmap, cb * BK, wx, hy, u.n, 0, &sh.full[s]);  // [hi][lo] x BN rows
                } else {
                    // pixel chunk c of shard r: (n, BK-column piece, ho), rows fastest so the
                    // taps of one column strip reuse its rows while they are still in L2; the
                    // tap's column shift s = v - pad is read from the copy shifted right by
                    // jc = (-s) mod 4
                    const int qa = u.r / p.Sw, qb = u.r - qa * p.Sw;  // row and column shard
                    const int ho = qa * p.own_h + (int)(c % p.own_h);
                    const long long rest = c / p.own_h;
                    const int wc = (int)(rest % p.row_chunks), n = (int)(rest / p.row_chunks);
                    const int w = qb * p.own_w + wc * BK;
                    tma_5d(st, &amap, w, u.m0, ho, n, 0, &sh.full[s]);  // [hi][lo] x 128 rows
                    // B = the hi rows of both slots, then their lo rows (one N = 256 operand
                    // pair); a slot is (tap, 128-channel block); the copy index jc and the
                    // image index share one box dimension (jc * N + n), hi / lo is the last
                    for (int h = 0; h < 2; h++) {
                        const int slot = 2 * u.tap + h;
                        if (slot >= p.slots) break;
                        const int tap = slot / p.nblocks, ci0 = (slot % p.nblocks) * 128;
                        const int uu = tap / p.kw, sft = tap % p.kw - p.pad;
                        const int jc = ((-sft) % 4 + 4) % 4;
                        unsigned char* dst = st + 2 * a_bytes + (uint32_t)h * WG_SLOT_BYTES;
                        tma_5d(dst, &bmap, w + sft + jc, ci0, ho + uu - p.pad, jc * p.N + n, 0, &sh.full[s]);
                        tma_5d(dst + b_bytes, &bmap, w + sft + jc, ci0, ho + uu - p.pad, jc * p.N + n, 1, &sh.full[s]);
                    }
                }
            }
        }
        if (*abort_flag) {
            // wait (bounded, ignoring the abort flag) for the last copy issued into each stage
            int zero = 0;
            for (long long k = it - p.stages > 0 ? it - p.stages : 0; k < it; k++)
                mbar_wait(&sh.full[k % p.stages], (unsigned)((k / p.stages) & 1), &zero);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        long long it = 0;
        long long g = 0;  // group counter = TMEM buffer position
        bool ok = true;
        for (int t = blockIdx.x; t < p.units && ok && !*abort_flag; t += gridDim.x) {
            const Unit u = decode(p, t, BN);
            uint32_t idesc = idesc_tf32(BM, BN, 0, 0);
            if (FMT == 1) {
                // a bf16 weight-gradient pair without a second slot: N = its real channels
                // (rounded up to 16), e.g. 48 for a 4x4/s4 conv over 3 channels
                int ncol = BN;
                if (p.mode == 1 && 2 * u.tap + 1 >= p.slots) {
                    const int kv = p.kvalid - 2 * u.tap * WG_SLOT;
                    ncol = kv >= WG_SLOT ? WG_SLOT : (kv + 15) / 16 * 16;
                }
                idesc = idesc_bf16(BM, ncol, 0, p.mode == 0 ? 1 : 0);
            }
            for (long long c0 = u.c_begin; c0 < u.c_end && ok; c0 += p.group, g++) {
                const int b = (int)(g & 1);
                if (g >= 2 && !mbar_wait(&sh.buf_empty[b], (unsigned)(((g >> 1) - 1) & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * 256);
                const long long c1 = c0 + p.group < u.c_end ? c0 + p.group : u.c_end;
                bool first = true;
                bool first_slot[2] = {true, true};
                for (long long c = c0; c < c1; c++, it++) {
                    const int s = (int)(it % p.stages);
                    if (!mbar_wait(&sh.full[s], (unsigned)((it / p.stages) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (FMT == 1 && p.bmn) {
                        // A as in the 1x1 weight gradient; B per slot: MN-major, 128-byte swizzle,
                        // two 64-channel blocks BKH rows apart, 8-pixel groups 1 KB apart, the
                        // three pieces a third of the slot apart.  Slot h accumulates into TMEM
                        // columns 128 h .. 128 h + 127 (N = 128).
                        constexpr int kPa[6] = {1, 2, 0, 1, 0, 0}, kPb[6] = {1, 0, 2, 0, 1, 0};
                        unsigned char* st = ring + (size_t)s * p.stage_bytes;
                        const uint64_t a0 = sdesc(st, 16, 512, 4);
                        const uint32_t ap = (uint32_t)p.a_piece >> 4, pb = (uint32_t)(p.b_piece / 2) >> 4;
                        const int slot_bytes = 3 * (p.b_piece / 2);
                        const int nsl = 2 * u.tap + 1 < p.slots ? 2 : 1;
                        const uint32_t id128 = idesc_bf16(BM, 128, 0, 1);
#pragma unroll
                        for (int k = 0; k < BKH / 16; k++) {
#pragma unroll
                            for (int t = 0; t < 6; t++) {
#pragma unroll
                                for (int h = 0; h < 2; h++) {
                                    if (h >= nsl) break;
                                    const uint64_t b0 = sdesc(st + 3 * p.a_piece + h * slot_bytes, BKH * 128, 1024, 2);
                                    tc_mma_bf16(d + (uint32_t)(128 * h), a0 + kPa[t] * ap + 2 * k,
                                                b0 + kPb[t] * pb + k * (2048 >> 4), id128, first_slot[h] ? 0u : 1u);
                                    first_slot[h] = false;
                                }
                            }
                        }
                        tc_commit(&sh.empty[s]);
                        continue;
                    }
                    if (FMT == 1) {
                        // A: K-major, 64-byte swizzle, 8-row groups 512 B apart (both modes).  B:
                        // conv mode MN-major, 128-byte swizzle, 64-pixel blocks BKH rows apart and
                        // 8-channel groups 1 KB apart; wgrad mode K-major like A.  Products a_i*b_j
                        // with i + j <= 2, the small ones first
                        // (offsets are added to the descriptors' start field, in 16-byte units)
                        constexpr int kPa[6] = {1, 2, 0, 1, 0, 0}, kPb[6] = {1, 0, 2, 0, 1, 0};
                        unsigned char* st = ring + (size_t)s * p.stage_bytes;
                        const uint64_t a0 = sdesc(st, 16, 512, 4);
                        const uint64_t b0 = p.mode == 0 ? sdesc(st + 3 * p.a_piece, BKH * 128, 1024, 2)
                                                        : sdesc(st + 3 * p.a_piece, 16, 512, 4);
                        const uint32_t ap = (uint32_t)p.a_piece >> 4, bp = (uint32_t)p.b_piece >> 4;
                        const uint32_t bk = p.mode == 0 ? 2048 >> 4 : 32 >> 4;
#pragma unroll
                        for (int k = 0; k < BKH / 16; k++) {  // 16 bf16 per MMA
#pragma unroll
                            for (int t = 0; t < 6; t++) {
                                tc_mma_bf16(d, a0 + kPa[t] * ap + 2 * k, b0 + kPb[t] * bp + k * bk, idesc,
                                            first ? 0u : 1u);
                                first = false;
                            }
                        }
                        tc_commit(&sh.empty[s]);
                        continue;
                    }
                    unsigned char* st = ring + (size_t)s * stage_bytes;
                    unsigned char *ahi = st, *alo = st + a_bytes, *bhi = st + 2 * a_bytes, *blo = bhi + b_bytes;
#pragma unroll
                    for (int k = 0; k < BK / 8; k++) {  // 8 tf32 = 32 bytes along the swizzled row
                        const uint64_t dah = sdesc(ahi + 32 * k, 16, SW_ATOM), dal = sdesc(alo + 32 * k, 16, SW_ATOM);
                        const uint64_t dbh = sdesc(bhi + 32 * k, 16, SW_ATOM), dbl = sdesc(blo + 32 * k, 16, SW_ATOM);
                        tc_mma(d, dal, dbh, idesc, first ? 0u : 1u);
                        tc_mma(d, dah, dbl, idesc, 1u);
                        tc_mma(d, dah, dbh, idesc, 1u);
                        first = false;
                    }
                    tc_commit(&sh.empty[s]);  // frees the stage once these MMAs have read it
                }
                if (ok) tc_commit(&sh.buf_full[b]);
            }
        }
        // every MMA issued has completed before tensor memory is released
        tc_commit(&sh.drain);
        int zero = 0;
        mbar_wait(&sh.drain, 0, &zero);
    } else if (warp >= 2) {
        // ---------------- epilogue ----------------
        const int ew = warp - 2;
        const int q = warp & 3;                // TMEM lane quarter this warp may access
        const int half = ew >> 2;              // column half
        const int row = 32 * q + lane;
        constexpr int HC = BN / 2;             // columns per thread
        long long g = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.units && ok && !*abort_flag; t += gridDim.x) {
            const Unit u = decode(p, t, BN);
            float acc[HC];
#pragma unroll
            for (int i = 0; i < HC; i++) acc[i] = 0.0f;
            for (long long c0 = u.c_begin; c0 < u.c_end; c0 += p.group, g++) {
                const int b = (int)(g & 1);
                if (!mbar_wait(&sh.buf_full[b], (unsigned)((g >> 1) & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * 256 + half * HC);
#pragma unroll
                for (int cc = 0; cc < HC; cc += 32) {
                    float v[32];
                    tc_ld32(base + (uint32_t)cc, v);
#pragma unroll
                    for (int i = 0; i < 32; i++) acc[cc + i] += v[i];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.buf_empty[b]);
            }
            if (!ok) break;
            if (p.mode == 0 && p.d2s) {
                // row m = (uu*C + c)*sd + vv holds image pixels (ho*sd + uu, (w0 + k)*sd + vv)
                const int m = u.m0 + row, sd = p.d2s;
                const bool valid = m < sd * sd * p.d2s_c;
                const int uc = m / sd, vv = m - uc * sd, uu = uc / p.d2s_c, c = uc - uu * p.d2s_c;
                const int Wimg = p.Wo * sd;
                float* dst = p.out + (((long long)u.n * p.d2s_c + c) * p.Ho * sd + u.ho * sd + uu) * Wimg +
                             (long long)(u.w0 + half * HC) * sd;
                if (sd == 2) {
                    // lanes 2i, 2i+1 hold vv = 0, 1 of one (uu, c) (s*s*C is even, so both or
                    // neither are valid); per 4 columns each passes the other two values and
                    // stores 4 consecutive pixels: lane vv=0 pixels 8j..8j+3, vv=1 8j+4..8j+7
                    const bool odd = vv != 0;
                    const unsigned mask = __activemask();  // the whole warp unless a wait timed out
#pragma unroll
                    for (int j = 0; j < HC / 4; j++) {
                        const float s0 = odd ? acc[4 * j] : acc[4 * j + 2];
                        const float s1 = odd ? acc[4 * j + 1] : acc[4 * j + 3];
                        const float r0 = __shfl_xor_sync(mask, s0, 1);
                        const float r1 = __shfl_xor_sync(mask, s1, 1);
                        const float4 o = odd ? make_float4(r0, acc[4 * j + 2], r1, acc[4 * j + 3])
                                             : make_float4(acc[4 * j], r0, acc[4 * j + 1], r1);
                        if (valid) *reinterpret_cast<float4*>(dst + 8 * j + (odd ? 4 : 0)) = o;
                    }
                } else if (valid) {
#pragma unroll
                    for (int k = 0; k < HC; k++) dst[(long long)k * sd + vv] = acc[k];
                }
            } else if (p.mode == 0 && p.tma_store) {
                // 32 columns at a time: the warp's 32 rows x 32 columns go to its staging
                // box (row = lane, 16-byte chunk j at j ^ (lane & 7): the 128-byte swizzle,
                // conflict-free per 8 lanes), then one lane stores the box with TMA
                const float bv = p.bias ? __ldg(p.bias + u.m0 + row) : 0.0f;
                unsigned char* box = stage_out + ew * TC_STAGE_OUT;
#pragma unroll
                for (int k = 0; k < HC / 32; k++) {
                    if (lane == 0) bulk_wait_read();  // the previous box has left shared memory
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        const int c = 32 * k + 4 * j;
                        *reinterpret_cast<float4*>(box + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                            make_float4(acc[c] + bv, acc[c + 1] + bv, acc[c + 2] + bv, acc[c + 3] + bv);
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&ymap, box, u.w0 + half * HC + 32 * k, u.ho, u.n * p.M + u.m0 + 32 * q);
                        bulk_commit();
                    }
                }
            } else if (p.mode == 0) {
                const int m = u.m0 + row;
                const float bv = p.bias ? __ldg(p.bias + m) : 0.0f;
                float* dst = p.out + (((long long)u.n * p.M + m) * p.Ho + u.ho) * p.Wo + u.w0 + half * HC;
#pragma unroll
                for (int k = 0; k < HC; k += 4)
                    *reinterpret_cast<float4*>(dst + k) =
                        make_float4(acc[k] + bv, acc[k + 1] + bv, acc[k + 2] + bv, acc[k + 3] + bv);
            } else {
                // column half = slot 2*pair + half (HC = 128 columns = one slot)
                const int slot = 2 * u.tap + half;
                if (slot < p.slots) {
                    const int tap = slot / p.nblocks, ci0 = (slot % p.nblocks) * 128;
                    const int co = u.m0 + row;
                    float* dst =
                        p.part + ((((long long)u.r * p.J + u.j) * p.taps + tap) * p.Co + co) * p.Ci + ci0;
#pragma unroll
                    for (int k = 0; k < HC; k += 4)
                        *reinterpret_cast<float4*>(dst + k) = make_float4(acc[k], acc[k + 1], acc[k + 2], acc[k + 3]);
                }
            }
        }
    }
    if (warp >= 2 && lane == 0 && p.tma_store) bulk_wait_all();  // output boxes written out
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tc_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// Operand preparation.
__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// NCHW [N][C][H][W] -> NHWC [N][H][W][Cp] split into tf32 hi / lo (channels
// C..Cp-1 zero).  Tiles of 64 channels x 32 columns go through shared memory
// (row pitch 33): 16-byte loads along the rows and 16-byte stores of four
// channels, both coalesced and free of bank conflicts.  Needs W % 4 == 0 and
// Cp % 64 == 0; 256 threads.
__global__ void __launch_bounds__(256) prep_nhwc_kernel(const float* __restrict__ x, float* __restrict__ hi,
                                                        float* __restrict__ lo, int C, int H, int W, int Cp) {
    __shared__ float t[64][33];
    const int w0 = blockIdx.x * 32, c0 = blockIdx.y * 64;
    const int nh = blockIdx.z;  // n * H + h
    const int n = nh / H, h = nh % H;
    const int tid = threadIdx.x;
#pragma unroll
    for (int it = 0; it < 2; it++) {  // 64 channel rows x 8 float4
        const int cl = tid / 8 + 32 * it, w4 = tid % 8;
        const int c = c0 + cl, w = w0 + 4 * w4;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (c < C && w < W) v = __ldg(reinterpret_cast<const float4*>(x + (((long long)n * C + c) * H + h) * W + w));
        t[cl][4 * w4] = v.x;
        t[cl][4 * w4 + 1] = v.y;
        t[cl][4 * w4 + 2] = v.z;
        t[cl][4 * w4 + 3] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 2; it++) {  // 32 pixels x 16 groups of four channels
        const int cg = tid % 8 + 8 * it, wl = tid / 8;
        const int w = w0 + wl;
        if (w < W) {
            const float4 v = make_float4(t[4 * cg][wl], t[4 * cg + 1][wl], t[4 * cg + 2][wl], t[4 * cg + 3][wl]);
            float4 vh, vl;
            vh.x = tf32_rna(v.x); vl.x = tf32_rna(v.x - vh.x);
            vh.y = tf32_rna(v.y); vl.y = tf32_rna(v.y - vh.y);
            vh.z = tf32_rna(v.z); vl.z = tf32_rna(v.z - vh.z);
            vh.w = tf32_rna(v.w); vl.w = tf32_rna(v.w - vh.w);
            const long long o = (((long long)n * H + h) * W + w) * Cp + c0 + 4 * cg;
            *reinterpret_cast<float4*>(hi + o) = vh;
            *reinterpret_cast<float4*>(lo + o) = vl;
        }
    }
}
hc_status launch_prep_nhwc(const float* x, float* hi, float* lo, int N, int C, int H, int W, int Cp,
                           cudaStream_t st) {
    if (Cp % 64 || W % 4 || (long long)N * H > 65535) return HC_ERR_UNSUPPORTED;
    prep_nhwc_kernel<<<dim3(cdiv(W, 32), Cp / 64, N * H), 256, 0, st>>>(x, hi, lo, C, H, W, Cp);
    return launched("prep_nhwc_kernel", st);
}

// Weights as the A operand of the conv pass: A[m][(u*kw+v)*Kc + c], hi / lo.
//   forward:    m = co, c = ci, value w[co][ci][u][v]
//   grad_input: m = ci, c = co, value w[co][ci][kh-1-u][kw-1-v]
__global__ void prep_weight_kernel(const float* __restrict__ w, float* __restrict__ hi, float* __restrict__ lo,
                                   int Co, int Ci, int kh, int kw, int Mp, int Kc, int transpose) {
    const long long ktot = (long long)kh * kw * Kc;
    const long long total = (long long)Mp * ktot;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(q / ktot);
        const int k = (int)(q % ktot);
        const int tap = k / Kc, c = k % Kc;
        const int u = tap / kw, v = tap % kw;
        float val = 0.0f;
        if (!transpose) {
            if (m < Co && c < Ci) val = __ldg(w + (((long long)m * Ci + c) * kh + u) * kw + v);
        } else {
            if (m < Ci && c < Co) val = __ldg(w + (((long long)c * Ci + m) * kh + (kh - 1 - u)) * kw + (kw - 1 - v));
        }
        const float vh = tf32_rna(val);
        hi[q] = vh;
        lo[q] = tf32_rna(val - vh);
    }
}

// NCHW -> NCHW tf32 hi / lo (the grad_output operand of the weight gradient).
// tf32 hi / lo split of an NCHW tensor, stored row-interleaved as [N][H][C][W]:
// the C rows of one image row sit together, so a TMA box of many channels x a
// few pixels covers a few hundred KB instead of one page per channel plane.
// Block (image row n*H + h, 16 channels): 16 input rows of W floats, read and
// written as contiguous float4 runs.  Needs W % 4 == 0; 256 threads.
__global__ void __launch_bounds__(256) prep_split_rows_kernel(const float* __restrict__ x, float* __restrict__ hi,
                                                              float* __restrict__ lo, int C, int H, int W) {
    const int nh = blockIdx.x, n = nh / H, h = nh - n * H;
    const int c0 = blockIdx.y * 16, nc = C - c0 < 16 ? C - c0 : 16;
    const int W4 = W / 4, items = nc * W4;
    const float4* src = reinterpret_cast<const float4*>(x) + (((long long)n * C + c0) * H + h) * W4;
    const long long o0 = ((long long)nh * C + c0) * W4;
    const long long plane4 = (long long)H * W4;
    for (int i = threadIdx.x; i < items; i += 256) {
        const int cl = i / W4, j = i - cl * W4;
        const float4 v = __ldg(src + cl * plane4 + j);
        float4 hv, l;
        hv.x = tf32_rna(v.x); l.x = tf32_rna(v.x - hv.x);
        hv.y = tf32_rna(v.y); l.y = tf32_rna(v.y - hv.y);
        hv.z = tf32_rna(v.z); l.z = tf32_rna(v.z - hv.z);
        hv.w = tf32_rna(v.w); l.w = tf32_rna(v.w - hv.w);
        reinterpret_cast<float4*>(hi)[o0 + i] = hv;
        reinterpret_cast<float4*>(lo)[o0 + i] = l;
    }
}
hc_status launch_split_rows(const float* x, float* hi, float* lo, int N, int C, int H, int W, cudaStream_t st) {
    if (W % 4 || (long long)N * H > 0x7fffffffLL || (C + 15) / 16 > 65535) return HC_ERR_UNSUPPORTED;
    prep_split_rows_kernel<<<dim3((unsigned)(N * H), (C + 15) / 16), 256, 0, st>>>(x, hi, lo, C, H, W);
    return launched("prep_split_rows_kernel", st);
}

// Space-to-depth for a k = stride = s convolution without padding (each output
// pixel reads one s x s block): channel k = (u*s + v)*C + c of output pixel
// (ho, wo) is x[c][ho*s + u][wo*s + v]; channels k >= s*s*C are zero.
//   NHWC form [N][Ho][Wo][Kp] (the forward's B operand), tf32 hi / lo.  Block
//   (32 output columns, 32 channels, (n, ho)): for each kernel row u the 32
//   input rows are staged in shared memory (coalesced reads), then written as
//   32 consecutive channels per (wo, v) (coalesced writes).
__global__ void prep_s2d_nhwc_kernel(const float* __restrict__ x, float* __restrict__ hi, float* __restrict__ lo,
                                     int C, int H, int W, int s, int Kp) {
    __shared__ float t[32][4 * 32 + 1];
    const int Ho = H / s, Wo = W / s;
    const int wo0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
    const int n = blockIdx.z / Ho, ho = blockIdx.z % Ho;
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int cols = 32 * s;
    for (int u = 0; u < s; u++) {
        for (int i = ty; i < 32; i += blockDim.y) {
            const int c = c0 + i;
            for (int col = tx; col < cols; col += 32) {
                const int w = wo0 * s + col;
                t[i][col] = (c < C && w < W) ? __ldg(x + (((long long)n * C + c) * H + ho * s + u) * W + w) : 0.0f;
            }
        }
        __syncthreads();
        for (int i = ty; i < 32; i += blockDim.y) {
            const int wo = wo0 + i, c = c0 + tx;
            if (wo < Wo && c < C) {
                for (int v = 0; v < s; v++) {
                    const float val = t[tx][i * s + v];
                    const float h = tf32_rna(val);
                    const long long o = (((long long)n * Ho + ho) * Wo + wo) * Kp + (u * s + v) * C + c;
                    hi[o] = h;
                    lo[o] = tf32_rna(val - h);
                }
            }
        }
        __syncthreads();
    }
}
// The same for C % 64 == 0, with 16-byte accesses: block (32 output columns,
// 64 channels, (n, ho)), 256 threads, shared tile [64][32*S + 1].  For each
// kernel row u the 64 input rows are read as float4 (coalesced), then every
// (input column, four channels) is written as one float4 to output pixel
// wo = col / S, channel block v = col % S (128 contiguous bytes per 8 lanes;
// 8 channel groups x 4 columns per warp hit 32 distinct banks).
template <int S>
__global__ void __launch_bounds__(256) prep_s2d_nhwc64_kernel(const float* __restrict__ x, float* __restrict__ hi,
                                                              float* __restrict__ lo, int C, int H, int W, int Kp) {
    extern __shared__ float t2[];  // [64][32 * S + 1]
    constexpr int COLS = 32 * S, PITCH = COLS + 1;
    const int Ho = H / S, Wo = W / S;
    const int wo0 = blockIdx.x * 32, c0 = blockIdx.y * 64;
    const int n = blockIdx.z / Ho, ho = blockIdx.z % Ho;
    const int tid = threadIdx.x;
#pragma unroll 1
    for (int u = 0; u < S; u++) {
#pragma unroll
        for (int i = 0; i < 2 * S; i++) {  // 64 rows x 8*S float4
            const int idx = tid + 256 * i;
            const int cl = idx / (8 * S), q = idx % (8 * S);
            const int w = wo0 * S + 4 * q;
            float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (w < W)
                v = __ldg(reinterpret_cast<const float4*>(x + (((long long)n * C + c0 + cl) * H + ho * S + u) * W + w));
            float* r = t2 + cl * PITCH + 4 * q;
            r[0] = v.x;
            r[1] = v.y;
            r[2] = v.z;
            r[3] = v.w;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 2 * S; i++) {  // COLS columns x 16 groups of four channels
            const int idx = tid + 256 * i;
            const int cg = idx % 8 + 8 * (idx / (8 * COLS));
            const int col = (idx / 8) % COLS;
            const int wo = wo0 + col / S, v = col % S;
            if (wo < Wo) {
                const float* r = t2 + 4 * cg * PITCH + col;
                const float4 a = make_float4(r[0], r[PITCH], r[2 * PITCH], r[3 * PITCH]);
                float4 vh, vl;
                vh.x = tf32_rna(a.x); vl.x = tf32_rna(a.x - vh.x);
                vh.y = tf32_rna(a.y); vl.y = tf32_rna(a.y - vh.y);
                vh.z = tf32_rna(a.z); vl.z = tf32_rna(a.z - vh.z);
                vh.w = tf32_rna(a.w); vl.w = tf32_rna(a.w - vh.w);
                const long long o = (((long long)n * Ho + ho) * Wo + wo) * Kp + (u * S + v) * C + c0 + 4 * cg;
                *reinterpret_cast<float4*>(hi + o) = vh;
                *reinterpret_cast<float4*>(lo + o) = vl;
            }
        }
        __syncthreads();
    }
}
// The same for few input channels (s*s*C <= 512, C % 64 != 0; the stem's C = 3):
// block (32 output columns, (n, ho)), 256 threads.  The C*S input rows of the
// block's s x s windows (32*S floats each) are staged in shared memory as
// float4s; then each warp writes whole output pixels, lane l the channel groups
// 4l, 4l + 128, ... of Kp, zeros past s*s*C included (512 contiguous bytes per
// 128 channels, hi and lo).
template <int S>
__global__ void __launch_bounds__(256) prep_s2d_nhwc_small_kernel(const float* __restrict__ x, float* __restrict__ hi,
                                                                  float* __restrict__ lo, int C, int H, int W,
                                                                  int Kp) {
    extern __shared__ float t3[];  // [C][S][32*S]
    constexpr int COLS = 32 * S;
    const int Ho = H / S, Wo = W / S;
    const int wo0 = blockIdx.x * 32;
    const int n = blockIdx.y / Ho, ho = blockIdx.y % Ho;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q4 = C * S * (COLS / 4);
    for (int i = tid; i < q4; i += 256) {
        const int r = i / (COLS / 4), q = i - r * (COLS / 4);  // r = c*S + u
        const int c = r / S, u = r - c * S;
        const int w = wo0 * S + 4 * q;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (w < W) v = __ldg(reinterpret_cast<const float4*>(x + (((long long)n * C + c) * H + ho * S + u) * W + w));
        float* d = t3 + r * COLS + 4 * q;
        d[0] = v.x;
        d[1] = v.y;
        d[2] = v.z;
        d[3] = v.w;
    }
    __syncthreads();
    const int kreal = S * S * C;
    for (int pl = warp; pl < 32; pl += 8) {
        const int wo = wo0 + pl;
        if (wo >= Wo) break;
        const long long o = (((long long)n * Ho + ho) * Wo + wo) * Kp;
        for (int k0 = 4 * lane; k0 < Kp; k0 += 128) {
            float e[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int kk = k0 + j;
                float val = 0.0f;
                if (kk < kreal) {
                    const int tap = kk / C, c = kk - tap * C, u = tap / S, v = tap - u * S;
                    val = t3[(c * S + u) * COLS + pl * S + v];
                }
                e[j] = val;
            }
            float4 vh, vl;
            vh.x = tf32_rna(e[0]); vl.x = tf32_rna(e[0] - vh.x);
            vh.y = tf32_rna(e[1]); vl.y = tf32_rna(e[1] - vh.y);
            vh.z = tf32_rna(e[2]); vl.z = tf32_rna(e[2] - vh.z);
            vh.w = tf32_rna(e[3]); vl.w = tf32_rna(e[3] - vh.w);
            *reinterpret_cast<float4*>(hi + o + k0) = vh;
            *reinterpret_cast<float4*>(lo + o + k0) = vl;
        }
    }
}
// Zero the channel tail [k0, Kp) of every pixel of an NHWC hi / lo pair.
__global__ void zero_tail_kernel(float* __restrict__ hi, float* __restrict__ lo, long long pixels, int k0, int Kp) {
    const int tail = Kp - k0;
    const long long total = pixels * tail;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        const long long o = (q / tail) * Kp + k0 + q % tail;
        hi[o] = 0.0f;
        lo[o] = 0.0f;
    }
}
//   row-interleaved planar form [N][Ho][Kp][Wo] (the weight gradient's B
//   operand: pixels contiguous).  Each item reads 4*S consecutive columns of one
//   input row (n, c, h = ho*S + u) as S float4 and writes, for every v, the four
//   output columns wo = 4j..4j+3 of row (n, ho, (u*S + v)*C + c) as one float4.
//   Needs Wo % 4 == 0.
template <int S>
__global__ void prep_s2d_planar_kernel(const float* __restrict__ x, float* __restrict__ hi, float* __restrict__ lo,
                                       int C, int H, int W, int Kp, long long items) {
    const int Ho = H / S, Wo = W / S, J = Wo / 4;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < items;
         q += (long long)gridDim.x * blockDim.x) {
        const long long rid = q / J;  // (n * C + c) * H + h
        const int j = (int)(q - rid * J);
        const int h = (int)(rid % H);
        const long long nc = rid / H;
        const int c = (int)(nc % C);
        const long long n = nc / C;
        const int ho = h / S, u = h - ho * S;
        float e[4 * S];
        const float4* src = reinterpret_cast<const float4*>(x + rid * W + 4LL * j * S);
#pragma unroll
        for (int k = 0; k < S; k++) {
            const float4 a = __ldg(src + k);
            e[4 * k] = a.x;
            e[4 * k + 1] = a.y;
            e[4 * k + 2] = a.z;
            e[4 * k + 3] = a.w;
        }
#pragma unroll
        for (int v = 0; v < S; v++) {
            const float4 a = make_float4(e[v], e[S + v], e[2 * S + v], e[3 * S + v]);
            float4 vh, vl;
            vh.x = tf32_rna(a.x); vl.x = tf32_rna(a.x - vh.x);
            vh.y = tf32_rna(a.y); vl.y = tf32_rna(a.y - vh.y);
            vh.z = tf32_rna(a.z); vl.z = tf32_rna(a.z - vh.z);
            vh.w = tf32_rna(a.w); vl.w = tf32_rna(a.w - vh.w);
            const long long o = ((n * Ho + ho) * Kp + (u * S + v) * C + c) * Wo + 4LL * j;
            *reinterpret_cast<float4*>(hi + o) = vh;
            *reinterpret_cast<float4*>(lo + o) = vl;
        }
    }
}
// Weights in space-to-depth order: forward A[co][k] = w[co][c][u][v] with
// k = (u*s + v)*C + c; grad_input (transpose) A[m][co] = w[co][c][u][v] with
// m = (u*C + c)*s + v, so that the s outputs of one (u, c) that interleave along
// an image row sit in adjacent TMEM lanes.  Rows / columns >= s*s*C are zero.
__global__ void prep_weight_s2d_kernel(const float* __restrict__ w, float* __restrict__ hi, float* __restrict__ lo,
                                       int Co, int C, int s, int Kp, int transpose) {
    const long long total = (long long)Co * Kp;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        int co, k;
        if (!transpose) {
            co = (int)(q / Kp);
            k = (int)(q % Kp);
        } else {
            k = (int)(q / Co);
            co = (int)(q % Co);
        }
        float v = 0.0f;
        if (k < s * s * C) {
            int c, uu, vv;
            if (!transpose) {  // k = (u*s + v)*C + c: the channel order of the space-to-depth copies
                const int tap = k / C;
                c = k - tap * C;
                uu = tap / s;
                vv = tap - uu * s;
            } else {  // row k = (u*C + c)*s + v: the s rows of one (u, c) are adjacent
                const int uc = k / s;
                vv = k - uc * s;
                uu = uc / C;
                c = uc - uu * C;
            }
            v = __ldg(w + (((long long)co * C + c) * s + uu) * s + vv);
        }
        const float h = tf32_rna(v);
        hi[q] = h;
        lo[q] = tf32_rna(v - h);
    }
}
// Weight-gradient partials in space-to-depth order back to [S][Co][C][s][s]:
// gwp[r][co][c][u][v] = sum_j part[r][j][co][(u*s + v)*C + c] (j ascending).
// One block per (r, co) row: threads walk k (coalesced reads), writes scatter.
__global__ void wgrad_reduce_s2d_kernel(const float* __restrict__ part, float* __restrict__ gwp, int J, int Co,
                                        int C, int s, int Kp) {
    const int r = blockIdx.x / Co, co = blockIdx.x - r * Co, K = s * s * C;
    const float* src = part + ((long long)r * J * Co + co) * Kp;
    float* dst = gwp + (long long)blockIdx.x * K;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        float t = 0.0f;
        for (int j = 0; j < J; j++) t += src[(long long)j * Co * Kp + k];
        const int tap = k / C, c = k - tap * C;  // tap = u*s + v
        dst[c * s * s + tap] = t;
    }
}

// Weight-gradient partials: gwp[r][co][ci][tap] = sum_j part[r][j][tap][co][ci]
// (j ascending).  One block per (r, co) row: threads walk ci (coalesced reads).
__global__ void wgrad_reduce_kernel(const float* __restrict__ part, float* __restrict__ gwp, int J, int taps,
                                    int Co, int Ci) {
    const int r = blockIdx.x / Co, co = blockIdx.x - r * Co;
    const long long per = (long long)taps * Co * Ci;
    float* dst = gwp + (long long)blockIdx.x * Ci * taps;
    for (int q = threadIdx.x; q < taps * Ci; q += blockDim.x) {
        const int tap = q / Ci, ci = q - tap * Ci;
        const float* src = part + (long long)r * J * per + ((long long)tap * Co + co) * Ci + ci;
        float t = 0.0f;
        for (int j = 0; j < J; j++) t += src[(long long)j * per];
        dst[ci * taps + tap] = t;
    }
}

// fp32 -> three bf16 pieces (split3, common.cuh), piece k of value i at
// out[k * ps + i].  Elementwise over n4 float4s (the layout is kept); ps4 =
// piece stride / 4.  MODE 1: the pieces of GELU(x); MODE 2: of x * GELU'(y)
// (gelu_f / gelu_d, common.cuh).
template <int MODE>
__global__ void __launch_bounds__(256) prep_pieces_kernel(const float4* __restrict__ x, const float4* __restrict__ y,
                                                          uint2* __restrict__ out, long long n4, long long ps4) {
    for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n4; i += (long long)gridDim.x * 256) {
        float4 v = __ldg(x + i);
        if (MODE == 1) v = make_float4(gelu_f(v.x), gelu_f(v.y), gelu_f(v.z), gelu_f(v.w));
        if (MODE == 2) {
            const float4 h = __ldg(y + i);
            v = make_float4(v.x * gelu_d(h.x), v.y * gelu_d(h.y), v.z * gelu_d(h.z), v.w * gelu_d(h.w));
        }
        store_pieces4(v, out, i, ps4);
    }
}
// Transposed pieces of a small R x C matrix: out[k * ps + c * R + r] = piece k of w[r * C + c].
__global__ void prep_pieces_t_kernel(const float* __restrict__ w, __nv_bfloat16* __restrict__ out, int R, int C,
                                     long long ps) {
    const long long i = blockIdx.x * 256LL + threadIdx.x;
    if (i >= (long long)R * C) return;
    const int c = (int)(i / R), r = (int)(i % R);
    __nv_bfloat16 a, b, e;
    split3(__ldg(w + (long long)r * C + c), a, b, e);
    out[i] = a;
    out[ps + i] = b;
    out[2 * ps + i] = e;
}

// x [N][C][H][W] -> three bf16 pieces in the channel-blocked NHWC layout
// [N][H][W][C/128][3][128]: piece k of channel c at pixel (n, h, w) is element
// (((n*H + h)*W + w)*(C/128) + c/128)*384 + k*128 + c%128 -- the weight
// gradient's B operand, where a tap's pixel shift is a plain TMA coordinate.
// A block takes 32 columns of one row (n, h) and walks the 128-channel blocks:
// 128 rows x 32 floats through shared memory (16-byte loads along the rows,
// pitch 33: no bank conflicts either way), then each thread splits 16 channels
// of one pixel and writes 32 contiguous bytes per piece.  Needs C % 128 == 0
// and W % 4 == 0; 256 threads.
__global__ void __launch_bounds__(256) prep_pieces_nhwc_kernel(const float* __restrict__ x,
                                                               __nv_bfloat16* __restrict__ out, int C, int H, int W) {
    __shared__ float t[128][33];
    const int tiles = (W + 31) / 32;
    const long long nh = blockIdx.x / tiles;
    const int w0 = (int)(blockIdx.x - nh * tiles) * 32;
    const int n = (int)(nh / H), h = (int)(nh - (long long)n * H);
    const int tid = threadIdx.x, wl = tid & 31, g = tid >> 5;
    const int blocks = C / 128;
    for (int cb = 0; cb < blocks; cb++) {
#pragma unroll
        for (int it = 0; it < 4; it++) {  // 128 channel rows x 8 float4
            const int cl = tid / 8 + 32 * it, w4 = tid % 8;
            const int c = cb * 128 + cl, w = w0 + 4 * w4;
            float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (w < W) v = __ldg(reinterpret_cast<const float4*>(x + (((long long)n * C + c) * H + h) * W + w));
            t[cl][4 * w4] = v.x;
            t[cl][4 * w4 + 1] = v.y;
            t[cl][4 * w4 + 2] = v.z;
            t[cl][4 * w4 + 3] = v.w;
        }
        __syncthreads();
        const int w = w0 + wl;
        if (w < W) {
            uint32_t q[3][8];
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                __nv_bfloat16 a[3], b[3];
                split3(t[16 * g + i][wl], a[0], a[1], a[2]);
                split3(t[16 * g + i + 1][wl], b[0], b[1], b[2]);
#pragma unroll
                for (int k = 0; k < 3; k++) q[k][i / 2] = pack2(a[k], b[k]);
            }
            __nv_bfloat16* o = out + ((nh * W + w) * blocks + cb) * 384 + 16 * g;
#pragma unroll
            for (int k = 0; k < 3; k++) {
                uint4* d4 = reinterpret_cast<uint4*>(o + 128 * k);
                d4[0] = make_uint4(q[k][0], q[k][1], q[k][2], q[k][3]);
                d4[1] = make_uint4(q[k][4], q[k][5], q[k][6], q[k][7]);
            }
        }
        __syncthreads();
    }
}

// Space-to-depth pieces: x [N][C][H][W] -> [3][N][K][Ho][Wo] with K = S*S*C and
// channel k = (u*S + v)*C + c holding x[n][c][ho*S + u][wo*S + v].  Each item
// reads 4*S consecutive columns of one input row (n, c, h = ho*S + u) and
// writes, for every v, output columns 4j..4j+3 of channel (u*S + v)*C + c.
// Needs Wo % 4 == 0; ps4 = piece stride / 4.
template <int S>
__global__ void prep_s2d_pieces_kernel(const float* __restrict__ x, uint2* __restrict__ out, int C, int H, int W,
                                       long long items, long long ps4) {
    const int Ho = H / S, Wo = W / S, J = Wo / 4, K = S * S * C;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < items;
         q += (long long)gridDim.x * blockDim.x) {
        const long long rid = q / J;  // (n * C + c) * H + h
        const int j = (int)(q - rid * J);
        const int h = (int)(rid % H);
        const long long nc = rid / H;
        const int c = (int)(nc % C);
        const long long n = nc / C;
        const int ho = h / S, u = h - ho * S;
        float e[4 * S];
        const float4* src = reinterpret_cast<const float4*>(x + rid * W + 4LL * j * S);
#pragma unroll
        for (int k = 0; k < S; k++) {
            const float4 a = __ldg(src + k);
            e[4 * k] = a.x;
            e[4 * k + 1] = a.y;
            e[4 * k + 2] = a.z;
            e[4 * k + 3] = a.w;
        }
#pragma unroll
        for (int v = 0; v < S; v++) {
            __nv_bfloat16 a[4], b[4], g[4];
#pragma unroll
            for (int t = 0; t < 4; t++) split3(e[t * S + v], a[t], b[t], g[t]);
            const long long o4 = (((n * K + (u * S + v) * C + c) * Ho + ho) * Wo + 4LL * j) / 4;
            out[o4] = make_uint2(pack2(a[0], a[1]), pack2(a[2], a[3]));
            out[ps4 + o4] = make_uint2(pack2(b[0], b[1]), pack2(b[2], b[3]));
            out[2 * ps4 + o4] = make_uint2(pack2(g[0], g[1]), pack2(g[2], g[3]));
        }
    }
}
// Weight pieces in space-to-depth order, K = s*s*C: forward A[co][k] = w[co][c][u][v]
// with k = (u*s + v)*C + c ([Co][K]); grad_input A[m][co] = w[co][c][u][v] with
// m = (u*C + c)*s + v ([K][Co]), the row order of the depth-to-space store.
__global__ void prep_weight_s2d_pieces_kernel(const float* __restrict__ w, __nv_bfloat16* __restrict__ out, int Co,
                                              int C, int s, int transpose, long long ps) {
    const int K = s * s * C;
    const long long q = blockIdx.x * 256LL + threadIdx.x;
    if (q >= (long long)Co * K) return;
    int co, k, c, uu, vv;
    if (!transpose) {
        co = (int)(q / K);
        k = (int)(q % K);
        const int tap = k / C;
        c = k - tap * C;
        uu = tap / s;
        vv = tap - uu * s;
    } else {
        k = (int)(q / Co);
        co = (int)(q % Co);
        const int uc = k / s;
        vv = k - uc * s;
        uu = uc / C;
        c = uc - uu * C;
    }
    __nv_bfloat16 a, b, g;
    split3(__ldg(w + (((long long)co * C + c) * s + uu) * s + vv), a, b, g);
    out[q] = a;
    out[ps + q] = b;
    out[2 * ps + q] = g;
}


// Accumulator columns of a conv-pass tile: a segment of one output row.  Every
// output pixel's sum over taps and channel chunks runs in the same order
// whichever tile holds it, and the boxes' neighbour-column reads at a shard
// edge are exactly that shard's halo, so a tile may cross shard boundaries;
// its width is picked from the whole row.
int pick_bn(int out_w) {
    if (out_w % 256 == 0) return 256;
    if (out_w % 128 == 0) return 128;
    return 0;
}

// Trace name of a tc_conv_kernel launch: operand format and pass.
const char* tc_pass_name(const TcParams& p) {
    if (p.fmt == 1) return p.mode == 1 ? "tc_conv_kernel bf16x6 weight-gradient pass" : "tc_conv_kernel bf16x6 conv pass";
    return p.mode == 1 ? "tc_conv_kernel 3xTF32 weight-gradient pass" : "tc_conv_kernel 3xTF32 conv pass";
}

template <int BN, int FMT>
hc_status launch_bn(const CUtensorMap& amap, const CUtensorMap& bmap, const CUtensorMap& ymap, TcParams p,
                    cudaStream_t st) {
    static std::atomic<unsigned long long> attr{0};
    once_per_device(attr, [&] {
        return cudaFuncSetAttribute(tc_conv_kernel<BN, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    TC_SMEM_MAX) == cudaSuccess;
    });
    int smem;
    if (p.fmt == 1) {
        // three pieces of A (128 x BKH) and B (BN x BKH) per stage; as many stages as
        // fit before the output boxes (conv mode: 2 for BN = 256) or in the whole
        // buffer (weight gradient: 3)
        p.a_piece = BM * BKH * 2;
        p.b_piece = BN * BKH * 2;
        p.stage_bytes = 3 * (p.a_piece + p.b_piece);
        p.stages = (p.tma_store ? TC_SMEM_RING : TC_SMEM_MAX - 1024) / p.stage_bytes;
        if (p.stages > 8) p.stages = 8;
        if (p.stages < 2) return HC_ERR_UNSUPPORTED;
        smem = p.tma_store ? TC_SMEM_MAX : p.stages * p.stage_bytes + 1024;
    } else {
        const int stage_bytes = 2 * BM * ROWB + 2 * BN * ROWB;
        p.stages = TC_SMEM_RING / stage_bytes;
        if (p.stages > 8) p.stages = 8;
        smem = TC_SMEM_MAX;
    }
    const int grid = p.units < device_sm_count() ? p.units : device_sm_count();
    tc_conv_kernel<BN, FMT><<<grid, TC_THREADS, smem, st>>>(amap, bmap, ymap, p);
    return launched(tc_pass_name(p), st);
}

// ymap: the conv-mode output as a TMA map (out_map); nullptr stores with plain
// per-thread writes (depth-to-space and weight-gradient passes).
hc_status launch_conv_pass(int BN, const CUtensorMap& amap, const CUtensorMap& bmap, TcParams p, cudaStream_t st,
                           const CUtensorMap* ymap = nullptr) {
    p.tma_store = ymap != nullptr;
    if (!ymap) ymap = &amap;  // unused
    p.group = 256 / BK;  // 256 k-values (96 MMAs) per TMEM accumulation group (BKH == BK)
    if (p.fmt == 1) {
        if (BN == 256) return launch_bn<256, 1>(amap, bmap, *ymap, p, st);
        if (BN == 128) return launch_bn<128, 1>(amap, bmap, *ymap, p, st);
    } else {
        if (BN == 256) return launch_bn<256, 0>(amap, bmap, *ymap, p, st);
        if (BN == 128) return launch_bn<128, 0>(amap, bmap, *ymap, p, st);
    }
    return HC_ERR_UNSUPPORTED;
}

// Every operand map covers a tf32 hi / lo pair (two equal arrays, lo - hi bytes
// apart) as its outermost dimension, so one box brings [hi][lo]: few large boxes
// keep the TMA unit's per-box cost low.
static hc_status pair_stride(const float* hi, const float* lo, uint64_t* stride) {
    const long long d = (const char*)lo - (const char*)hi;
    if (d <= 0 || d % 16) return HC_ERR_INVALID_ARG;
    *stride = (uint64_t)d;
    return HC_OK;
}
// NHWC activation map for the conv pass: dims (Cp, W, H, N, 2), box (BK, BN, 1, 1, 2).
hc_status act_map_conv(CUtensorMap* m, const float* hi, const float* lo, int N, int H, int W, int Cp, int BN) {
    uint64_t ps;
    if (hc_status e = pair_stride(hi, lo, &ps)) return e;
    const uint64_t dims[5] = {(uint64_t)Cp, (uint64_t)W, (uint64_t)H, (uint64_t)N, 2};
    const uint64_t strides[4] = {(uint64_t)Cp * 4, (uint64_t)W * Cp * 4, (uint64_t)H * W * Cp * 4, ps};
    const uint32_t box[5] = {BK, (uint32_t)BN, 1, 1, 2};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, hi, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
// Weight map: dims (Ktot, Mp, 2), box (BK, 128, 2).
hc_status weight_map(CUtensorMap* m, const float* hi, const float* lo, int Mp, long long ktot) {
    uint64_t ps;
    if (hc_status e = pair_stride(hi, lo, &ps)) return e;
    const uint64_t dims[3] = {(uint64_t)ktot, (uint64_t)Mp, 2};
    const uint64_t strides[2] = {(uint64_t)ktot * 4, ps};
    const uint32_t box[3] = {BK, 128, 2};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, hi, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
// NCHW output of a conv pass as TMA store boxes: dims (Wo, Ho, N*M), box (32, 1, 32):
// 32 output columns of one row for 32 channels.
hc_status out_map(CUtensorMap* m, float* base, int N, int M, int Ho, int Wo) {
    const uint64_t dims[3] = {(uint64_t)Wo, (uint64_t)Ho, (uint64_t)N * M};
    const uint64_t strides[2] = {(uint64_t)Wo * 4, (uint64_t)Ho * Wo * 4};
    const uint32_t box[3] = {32, 1, 32};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
// Row-interleaved [N][H][C][W] map for K-major weight-gradient tiles (pixels
// contiguous): dims (W, C, H, N, 2), box (BK, rows, 1, 1, 2): smem [hi][lo] x
// [rows channels][BK pixels].
hc_status rows_map(CUtensorMap* m, const float* hi, const float* lo, int N, int C, int H, int W, int rows) {
    uint64_t ps;
    if (hc_status e = pair_stride(hi, lo, &ps)) return e;
    const uint64_t dims[5] = {(uint64_t)W, (uint64_t)C, (uint64_t)H, (uint64_t)N, 2};
    const uint64_t strides[4] = {(uint64_t)W * 4, (uint64_t)C * W * 4, (uint64_t)H * C * W * 4, ps};
    const uint32_t box[5] = {BK, (uint32_t)rows, 1, 1, 2};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, hi, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
// Row-interleaved column-shifted copies [copies][N][H][C][Wc]: dims (Wc, C, H,
// copies * N, 2) (copy j of image n at j * N + n), box (BK, rows, 1, 1, 1): hi
// (coordinate 0) and lo (1) are loaded apart, into the hi and lo halves of B.
hc_status shifted_map(CUtensorMap* m, const float* hi, const float* lo, int N, int C, int H, int Wc, int rows,
                      int copies) {
    uint64_t ps;
    if (hc_status e = pair_stride(hi, lo, &ps)) return e;
    const uint64_t dims[5] = {(uint64_t)Wc, (uint64_t)C, (uint64_t)H, (uint64_t)copies * N, 2};
    const uint64_t strides[4] = {(uint64_t)Wc * 4, (uint64_t)C * Wc * 4, (uint64_t)H * C * Wc * 4, ps};
    const uint32_t box[5] = {BK, (uint32_t)rows, 1, 1, 1};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, hi, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// bf16 piece arrays: the three pieces of one tensor ps elements apart (the
// outermost map dimension), so one box brings all three.
// Weight pieces [3][M][K], K-major tiles of 128 rows x 32 k: dims (K, M, 3),
// box (32, 128, 3), 64-byte swizzle.
hc_status pieces_weight_map(CUtensorMap* m, const void* base, int M, int K, long long ps) {
    const uint64_t dims[3] = {(uint64_t)K, (uint64_t)M, 3};
    const uint64_t strides[2] = {(uint64_t)K * 2, (uint64_t)ps * 2};
    const uint32_t box[3] = {BKH, 128, 3};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}
// Activation pieces [3][N][C][P] (P pixels of an image, contiguous) as MN-major
// tiles of BN pixels x 32 channels: dims (64, C, P / 64, N, 3).  The 64-pixel
// block is a dimension of its own (stride 128 B) placed after the channel, so
// a box lands as [piece][pixel block][channel][64 pixels]: per pixel block, 32
// rows of 128 bytes with the 128-byte swizzle, the MN-major tile layout.
hc_status pieces_mn_map(CUtensorMap* m, const void* base, int N, int C, long long P, int BN, long long ps) {
    const uint64_t dims[5] = {64, (uint64_t)C, (uint64_t)(P / 64), (uint64_t)N, 3};
    const uint64_t strides[4] = {(uint64_t)P * 2, 128, (uint64_t)C * P * 2, (uint64_t)ps * 2};
    const uint32_t box[5] = {64, BKH, (uint32_t)(BN / 64), 1, 3};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}
// Pieces [3][N][C][H][W] as K-major tiles of `rows` channels x 32 pixels of one
// image row: dims (W, H, C, N, 3), box (32, 1, rows, 1, 3), 64-byte swizzle.
hc_status pieces_rows_map(CUtensorMap* m, const void* base, int N, int C, int H, int W, int rows, long long ps) {
    const uint64_t dims[5] = {(uint64_t)W, (uint64_t)H, (uint64_t)C, (uint64_t)N, 3};
    const uint64_t strides[4] = {(uint64_t)W * 2, (uint64_t)H * W * 2, (uint64_t)C * H * W * 2, (uint64_t)ps * 2};
    const uint32_t box[5] = {BKH, 1, (uint32_t)rows, 1, 3};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

// x pieces in the channel-blocked NHWC layout (prep_pieces_nhwc_kernel) as
// MN-major B tiles of one slot: dims (64, W, 6 * C/128, H, N) -- the third
// dimension walks the 64-channel blocks of a pixel, (128-channel block, piece,
// half) in that order, 128 bytes apart -- and box (64, 32, 6, 1, 1): for one
// pixel row segment of 32 columns, the slot's 128 channels in all three pieces,
// landing as [piece][64-channel half][32 pixels][64 channels] with the 128-byte
// swizzle.
hc_status pieces_nhwc_map(CUtensorMap* m, const void* base, int N, int C, int H, int W) {
    const uint64_t pix = (uint64_t)3 * C * 2;  // bytes per pixel
    const uint64_t dims[5] = {64, (uint64_t)W, (uint64_t)(6 * (C / 128)), (uint64_t)H, (uint64_t)N};
    const uint64_t strides[4] = {pix, 128, (uint64_t)W * pix, (uint64_t)H * W * pix};
    const uint32_t box[5] = {64, BKH, 6, 1, 1};
    return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

size_t al256(size_t b) { return (b + 255) & ~(size_t)255; }
// piece stride: the element count rounded up to 128 (256 bytes)
long long piece_stride(long long n) { return (n + 127) / 128 * 128; }

// gelu: split GELU(x); gelu_y: split x * GELU'(gelu_y) (same layout as x)
hc_status launch_prep_pieces(const float* x, void* out, long long n, long long ps, cudaStream_t st,
                             bool gelu = false, const float* gelu_y = nullptr) {
    if (n % 4 || ps % 4) return HC_ERR_UNSUPPORTED;
    long long blocks = (n / 4 + 255) / 256;
    if (blocks > 152LL * 16) blocks = 152LL * 16;
    if (blocks < 1) blocks = 1;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const float4* y4 = reinterpret_cast<const float4*>(gelu_y);
    uint2* o = reinterpret_cast<uint2*>(out);
    if (gelu_y)
        prep_pieces_kernel<2><<<(unsigned)blocks, 256, 0, st>>>(x4, y4, o, n / 4, ps / 4);
    else if (gelu)
        prep_pieces_kernel<1><<<(unsigned)blocks, 256, 0, st>>>(x4, nullptr, o, n / 4, ps / 4);
    else
        prep_pieces_kernel<0><<<(unsigned)blocks, 256, 0, st>>>(x4, nullptr, o, n / 4, ps / 4);
    return launched("prep_pieces_kernel", st);
}



// k = stride = s >= 2 without padding: every output pixel reads its own s x s
// block, so the conv is a 1x1 conv of the space-to-depth image.
bool is_s2d(const hc_conv_desc* d) {
    return d->groups == 1 && d->stride >= 2 && d->kh == d->stride && d->kw == d->stride && d->padding == 0;
}
int s2d_kp(const hc_conv_desc* d) { return (d->stride * d->stride * d->C_in + 127) / 128 * 128; }

}  // namespace

// ---------------------------------------------------------------------------
bool tc_supported(const hc_conv_desc* d, const Plan& p) {
    if (is_s2d(d)) {
        const int s = d->stride;
        return s <= 4 && d->C_out % BM == 0 && d->H % s == 0 && d->W % s == 0 && pick_bn(p.Wl / s) != 0 &&
               (p.Wl / s) % 32 == 0 && p.Wo == d->W / s && p.Ho == d->H / s;
    }
    if (d->groups != 1 || d->stride != 1 || d->kh != d->kw || d->padding != (d->kh - 1) / 2 || d->kh % 2 == 0)
        return false;
    if (d->C_out % BM || d->C_in % BM) return false;  // forward rows and grad_input rows in 128-blocks
    if (!pick_bn(p.Wl) || d->padding > 3) return false;
    if (p.Ho != d->H || p.Wo != d->W || d->W % 4) return false;
    return true;
}

int tc_wgrad_splits(const hc_conv_desc* d, const Plan& p) {
    const bool sd = is_s2d(d);
    const int KK = sd ? 1 : d->kh * d->kw;
    const int nb = sd ? s2d_kp(d) / WG_SLOT : d->C_in / WG_SLOT;
    const long long units0 = (long long)(d->C_out / BM) * ((KK * nb + 1) / 2) * p.Q;
    const long long chunks = (long long)d->N * p.Hlo * ((p.Wl / d->stride) / BK);
    // Units are equally long, so the persistent grid runs ceil(units / SMs) waves.
    // Take the smallest split that fills every SM and keeps the last wave at least
    // 95 % full (each unit at least 2048 pixels long); else the best-filled split.
    const long long P = device_sm_count();
    const long long jmax = chunks * BK / 2048 > 1 ? chunks * BK / 2048 : 1;
    long long best = 1;
    double best_fill = 0.0;
    for (long long J = 1; J <= jmax; J++) {
        const long long units = units0 * J;
        const double fill = (double)units / (double)(((units + P - 1) / P) * P);
        if (units >= P && fill >= 0.95) return (int)J;
        if (fill > best_fill + 1e-9) {
            best_fill = fill;
            best = J;
        }
    }
    return (int)best;
}

// Workspace: forward  [x NHWC hi][x NHWC lo][A hi][A lo]
//            backward [gy NHWC hi][lo][A' hi][lo][gy NHCW hi][lo][x shifted hi][lo][split-K partials]
size_t tc_ws_bytes(const hc_conv_desc* d, const Plan& p, int pass) {
    if (is_s2d(d)) {  // forward [s2d NHWC hi][lo][A hi][lo]; backward [gy NHWC hi][lo][A' hi][lo][gy NHCW hi][lo][s2d planar hi][lo][partials]
        const size_t npx = (size_t)d->N * p.Ho * p.Wo, kp = s2d_kp(d);
        const size_t ns = npx * kp, ng = npx * d->C_out, wsz = (size_t)d->C_out * kp;
        if (pass == 0) return 2 * al256(4 * ns) + 2 * al256(4 * wsz);
        const size_t part = al256(4 * (size_t)p.Q * tc_wgrad_splits(d, p) * wsz);
        return 4 * al256(4 * ng) + 2 * al256(4 * wsz) + 2 * al256(4 * ns) + part;
    }
    const int KK = d->kh * d->kw;
    const size_t nx = (size_t)d->N * d->C_in * d->H * d->W;
    const size_t ng = (size_t)d->N * d->C_out * p.Ho * p.Wo;
    const size_t wsz = (size_t)d->C_out * KK * d->C_in;
    if (pass == 0) return 2 * al256(4 * nx) + 2 * al256(4 * wsz);
    const int J = tc_wgrad_splits(d, p);
    const size_t part = al256(4 * (size_t)p.Q * J * wsz);
    return 2 * al256(4 * ng) + 2 * al256(4 * wsz) + al256(6 * (size_t)piece_stride((long long)ng)) +
           al256(6 * nx) + part;
}

static hc_status launch_prep_s2d_nhwc(const hc_conv_desc* d, const Plan& p, const float* x, float* hi, float* lo,
                                      int Kp, cudaStream_t st) {
    const int s = d->stride, C = d->C_in;
    if ((long long)d->N * p.Ho > 65535) return HC_ERR_UNSUPPORTED;
    const size_t small_smem = sizeof(float) * C * s * 32 * s;
    if (C % 64 && s * s * C <= 512 && small_smem <= 48 * 1024 && d->W % 4 == 0) {  // writes the zero tail too
        const dim3 grid(cdiv(p.Wo, 32), d->N * p.Ho);
        if (s == 2)
            prep_s2d_nhwc_small_kernel<2><<<grid, 256, small_smem, st>>>(x, hi, lo, C, d->H, d->W, Kp);
        else if (s == 3)
            prep_s2d_nhwc_small_kernel<3><<<grid, 256, small_smem, st>>>(x, hi, lo, C, d->H, d->W, Kp);
        else if (s == 4)
            prep_s2d_nhwc_small_kernel<4><<<grid, 256, small_smem, st>>>(x, hi, lo, C, d->H, d->W, Kp);
        else
            return HC_ERR_UNSUPPORTED;
        return launched("prep_s2d_nhwc_small_kernel", st);
    }
    if (C % 64 == 0 && d->W % 4 == 0) {
        const dim3 grid(cdiv(p.Wo, 32), C / 64, d->N * p.Ho);
        const size_t smem = sizeof(float) * 64 * (32 * s + 1);
        if (s == 2)
            prep_s2d_nhwc64_kernel<2><<<grid, 256, smem, st>>>(x, hi, lo, C, d->H, d->W, Kp);
        else if (s == 3)
            prep_s2d_nhwc64_kernel<3><<<grid, 256, smem, st>>>(x, hi, lo, C, d->H, d->W, Kp);
        else if (s == 4)
            prep_s2d_nhwc64_kernel<4><<<grid, 256, smem, st>>>(x, hi, lo, C, d->H, d->W, Kp);
        else
            return HC_ERR_UNSUPPORTED;
    } else {
        prep_s2d_nhwc_kernel<<<dim3(cdiv(p.Wo, 32), cdiv(C, 32), d->N * p.Ho), dim3(32, 8), 0, st>>>(x, hi, lo, C, d->H,
                                                                                                  d->W, s, Kp);
    }
    hc_status e = launched("prep_s2d_nhwc_kernel", st);
    if (e || Kp == s * s * C) return e;
    // the channel tail is a K range of the forward GEMM: it must hold zeros
    const long long pixels = (long long)d->N * p.Ho * p.Wo;
    zero_tail_kernel<<<152 * 16, 256, 0, st>>>(hi, lo, pixels, s * s * C, Kp);
    return launched("zero_tail_kernel", st);
}
static hc_status launch_prep_s2d_planar(const hc_conv_desc* d, const Plan& p, const float* x, float* hi, float* lo,
                                        int Kp, cudaStream_t st) {
    const int s = d->stride;
    if (p.Wo % 4) return HC_ERR_UNSUPPORTED;
    const long long items = (long long)d->N * d->C_in * d->H * (p.Wo / 4);
    long long blocks = (items + 255) / 256;
    if (blocks > 152LL * 32) blocks = 152LL * 32;
    if (blocks < 1) blocks = 1;
    if (s == 2)
        prep_s2d_planar_kernel<2><<<(unsigned)blocks, 256, 0, st>>>(x, hi, lo, d->C_in, d->H, d->W, Kp, items);
    else if (s == 3)
        prep_s2d_planar_kernel<3><<<(unsigned)blocks, 256, 0, st>>>(x, hi, lo, d->C_in, d->H, d->W, Kp, items);
    else if (s == 4)
        prep_s2d_planar_kernel<4><<<(unsigned)blocks, 256, 0, st>>>(x, hi, lo, d->C_in, d->H, d->W, Kp, items);
    else
        return HC_ERR_UNSUPPORTED;
    return launched("prep_s2d_planar_kernel", st);
}

static hc_status s2d_fwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* b,
                         float* y, void* ws, cudaStream_t st) {
    const int s = d->stride, Co = d->C_out, Kp = s2d_kp(d);
    const size_t ns = (size_t)d->N * p.Ho * p.Wo * Kp, wsz = (size_t)Co * Kp;
    char* q = (char*)ws;
    float* xh = (float*)q;
    q += al256(4 * ns);
    float* xl = (float*)q;
    q += al256(4 * ns);
    float* ah = (float*)q;
    q += al256(4 * wsz);
    float* al = (float*)q;
    if (s > 4) return HC_ERR_UNSUPPORTED;
    hc_status e = launch_prep_s2d_nhwc(d, p, x, xh, xl, Kp, st);
    if (e) return e;
    prep_weight_s2d_kernel<<<cdiv((long long)wsz, 256), 256, 0, st>>>(w, ah, al, Co, d->C_in, s, Kp, 0);
    if ((e = launched("prep_weight_s2d_kernel", st))) return e;
    const int BN = pick_bn(p.Wo);
    TcParams tp{};
    tp.mode = 0;
    tp.N = d->N;
    tp.Ho = p.Ho;
    tp.Wo = p.Wo;
    tp.M = Co;
    tp.Kc = Kp;
    tp.kh = 1;
    tp.kw = 1;
    tp.pad = 0;
    tp.tiles_w = p.Wo / BN;
    tp.mblocks = Co / BM;
    tp.chunks = Kp / BK;
    tp.units = tp.mblocks * d->N * p.Ho * tp.tiles_w;
    tp.bias = b;
    tp.out = y;
    CUtensorMap ma, mb, my;
    if ((e = weight_map(&ma, ah, al, Co, Kp)) || (e = act_map_conv(&mb, xh, xl, d->N, p.Ho, p.Wo, Kp, BN)) ||
        (e = out_map(&my, y, d->N, Co, p.Ho, p.Wo)))
        return e;
    return launch_conv_pass(BN, ma, mb, tp, st, &my);
}

static hc_status s2d_bwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* gy,
                         float* gx, float* gwp, bool want_w, void* ws, cudaStream_t st) {
    const int s = d->stride, Co = d->C_out, Ci = d->C_in, Kp = s2d_kp(d);
    const size_t npx = (size_t)d->N * p.Ho * p.Wo, ns = npx * Kp, ng = npx * Co, wsz = (size_t)Co * Kp;
    char* q = (char*)ws;
    float* gh = (float*)q;
    q += al256(4 * ng);
    float* gl = (float*)q;
    q += al256(4 * ng);
    float* ah = (float*)q;
    q += al256(4 * wsz);
    float* al = (float*)q;
    q += al256(4 * wsz);
    float* gch = (float*)q;
    q += al256(4 * ng);
    float* gcl = (float*)q;
    q += al256(4 * ng);
    float* sh = (float*)q;
    q += al256(4 * ns);
    float* sl = (float*)q;
    q += al256(4 * ns);
    float* part = (float*)q;
    const int BN = pick_bn(p.Wo);
    hc_status e;
    if (gx) {  // D[(u,v,c)][px] = sum_co w[co][c][u][v] gy[co][px], stored depth-to-space
        if ((e = launch_prep_nhwc(gy, gh, gl, d->N, Co, p.Ho, p.Wo, Co, st))) return e;
        prep_weight_s2d_kernel<<<cdiv((long long)wsz, 256), 256, 0, st>>>(w, ah, al, Co, Ci, s, Kp, 1);
        if ((e = launched("prep_weight_s2d_kernel", st))) return e;
        TcParams tp{};
        tp.mode = 0;
        tp.N = d->N;
        tp.Ho = p.Ho;
        tp.Wo = p.Wo;
        tp.M = Kp;
        tp.Kc = Co;
        tp.kh = 1;
        tp.kw = 1;
        tp.pad = 0;
        tp.tiles_w = p.Wo / BN;
        tp.mblocks = Kp / BM;
        tp.chunks = Co / BK;
        tp.units = tp.mblocks * d->N * p.Ho * tp.tiles_w;
        tp.out = gx;
        tp.d2s = s;
        tp.d2s_c = Ci;
        CUtensorMap ma, mb;
        if ((e = weight_map(&ma, ah, al, Kp, Co)) || (e = act_map_conv(&mb, gh, gl, d->N, p.Ho, p.Wo, Co, BN)))
            return e;
        if ((e = launch_conv_pass(BN, ma, mb, tp, st))) return e;
    }
    if (want_w) {  // G[co][(u,v,c)] = sum over a shard's pixels of gy[co][px] s2d[(u,v,c)][px]
        if ((e = launch_split_rows(gy, gch, gcl, d->N, Co, p.Ho, p.Wo, st))) return e;
        // channels k >= s*s*C of the planar copy are left unwritten: they are B rows,
        // i.e. accumulator columns of their own, which the reduction never reads
        if ((e = launch_prep_s2d_planar(d, p, x, sh, sl, Kp, st))) return e;
        TcParams tp{};
        tp.mode = 1;
        tp.Co = Co;
        tp.Ci = Kp;
        tp.S = p.Q;
        tp.Sw = p.S;
        tp.own_h = p.Hlo;
        tp.J = tc_wgrad_splits(d, p);
        tp.own_w = p.Wl / s;
        tp.row_chunks = tp.own_w / BK;
        tp.Ho = p.Ho;
        tp.kh = 1;
        tp.kw = 1;
        tp.pad = 0;
        tp.taps = 1;
        tp.mblocks = Co / BM;
        tp.nblocks = Kp / WG_SLOT;
        tp.slots = tp.nblocks;
        tp.shard_chunks = (long long)d->N * p.Hlo * tp.row_chunks;
        tp.units = tp.mblocks * ((tp.slots + 1) / 2) * tp.J * p.Q;
        tp.part = part;
        tp.N = d->N;
        CUtensorMap ma, mb;
        if ((e = rows_map(&ma, gch, gcl, d->N, Co, p.Ho, p.Wo, BM)) ||
            (e = shifted_map(&mb, sh, sl, d->N, Kp, p.Ho, p.Wo, WG_SLOT, 1)))
            return e;
        if ((e = launch_conv_pass(WG_BN, ma, mb, tp, st))) return e;
        wgrad_reduce_s2d_kernel<<<(unsigned)(p.Q * Co), 256, 0, st>>>(part, gwp, tp.J, Co, Ci, s, Kp);
        if ((e = launched("wgrad_reduce_s2d_kernel", st))) return e;
    }
    return HC_OK;
}

hc_status launch_tc_fwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* b,
                        float* y, void* ws, cudaStream_t st) {
    if (is_s2d(d)) return s2d_fwd(d, p, x, w, b, y, ws, st);
    const int K = d->kh, KK = K * K, Ci = d->C_in, Co = d->C_out;
    const size_t nx = (size_t)d->N * Ci * d->H * d->W, wsz = (size_t)Co * KK * Ci;
    char* q = (char*)ws;
    float* xh = (float*)q;
    q += al256(4 * nx);
    float* xl = (float*)q;
    q += al256(4 * nx);
    float* ah = (float*)q;
    q += al256(4 * wsz);
    float* al = (float*)q;
    hc_status s = launch_prep_nhwc(x, xh, xl, d->N, Ci, d->H, d->W, Ci, st);
    if (s) return s;
    prep_weight_kernel<<<cdiv((long long)wsz, 256), 256, 0, st>>>(w, ah, al, Co, Ci, K, K, Co, Ci, 0);
    if ((s = launched("prep_weight_kernel", st))) return s;
    const int BN = pick_bn(p.Wo);
    TcParams tp{};
    tp.mode = 0;
    tp.N = d->N;
    tp.Ho = p.Ho;
    tp.Wo = p.Wo;
    tp.M = Co;
    tp.Kc = Ci;
    tp.kh = K;
    tp.kw = K;
    tp.pad = d->padding;
    tp.tiles_w = p.Wo / BN;
    tp.mblocks = Co / BM;
    tp.chunks = KK * (Ci / BK);
    tp.units = tp.mblocks * d->N * p.Ho * tp.tiles_w;
    tp.bias = b;
    tp.out = y;
    CUtensorMap ma, mb, my;
    if ((s = weight_map(&ma, ah, al, Co, (long long)KK * Ci)) || (s = act_map_conv(&mb, xh, xl, d->N, d->H, d->W, Ci, BN)) ||
        (s = out_map(&my, y, d->N, Co, p.Ho, p.Wo)))
        return s;
    return launch_conv_pass(BN, ma, mb, tp, st, &my);
}

hc_status launch_tc_bwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* gy,
                        float* gx, float* gwp, bool want_w, void* ws, cudaStream_t st, float* gbp, float* btmp) {
    if (is_s2d(d)) return s2d_bwd(d, p, x, w, gy, gx, gwp, want_w, ws, st);
    const int K = d->kh, KK = K * K, Ci = d->C_in, Co = d->C_out;
    const size_t ng = (size_t)d->N * Co * p.Ho * p.Wo, wsz = (size_t)Co * KK * Ci;
    const size_t nx = (size_t)d->N * Ci * d->H * d->W;
    const long long psg = piece_stride((long long)ng);
    char* q = (char*)ws;
    float* gh = (float*)q;
    q += al256(4 * ng);
    float* gl = (float*)q;
    q += al256(4 * ng);
    float* ah = (float*)q;
    q += al256(4 * wsz);
    float* al = (float*)q;
    q += al256(4 * wsz);
    void* gp = q;  // grad_output's bf16 pieces [3][N][Co][Ho][Wo]
    q += al256(6 * (size_t)psg);
    __nv_bfloat16* xp = (__nv_bfloat16*)q;  // x's pieces [N][H][W][C/128][3][128]
    q += al256(6 * nx);
    float* part = (float*)q;
    hc_status s;
    if (gx) {  // grad_input = conv of grad_output with the flipped, transposed kernel
        if ((s = launch_prep_nhwc(gy, gh, gl, d->N, Co, p.Ho, p.Wo, Co, st))) return s;
        prep_weight_kernel<<<cdiv((long long)wsz, 256), 256, 0, st>>>(w, ah, al, Co, Ci, K, K, Ci, Co, 1);
        if ((s = launched("prep_weight_kernel", st))) return s;
        const int BN = pick_bn(p.Wo);
        TcParams tp{};
        tp.mode = 0;
        tp.N = d->N;
        tp.Ho = d->H;
        tp.Wo = d->W;
        tp.M = Ci;
        tp.Kc = Co;
        tp.kh = K;
        tp.kw = K;
        tp.pad = K - 1 - d->padding;
        tp.tiles_w = d->W / BN;
        tp.mblocks = Ci / BM;
        tp.chunks = KK * (Co / BK);
        tp.units = tp.mblocks * d->N * d->H * tp.tiles_w;
        tp.bias = nullptr;
        tp.out = gx;
        CUtensorMap ma, mb, my;
        if ((s = weight_map(&ma, ah, al, Ci, (long long)KK * Co)) ||
            (s = act_map_conv(&mb, gh, gl, d->N, p.Ho, p.Wo, Co, BN)) || (s = out_map(&my, gx, d->N, Ci, d->H, d->W)))
            return s;
        if ((s = launch_conv_pass(BN, ma, mb, tp, st, &my))) return s;
    }
    if (want_w) {
        // G[co][(tap, ci)] = sum over a shard's pixels of gy[co][px] x[ci][px + tap] on three
        // bf16 pieces per operand (six products, as the 1x1 convs): 16-bit operands may be
        // MN-major, so x's pieces stay in one NHWC copy and every tap's row and column shift
        // is a box coordinate.  The bias-gradient partials, when asked for, come from the
        // same read of grad_output as its pieces.
        if (gbp)
            s = launch_bias_grad_partials(gy, gbp, d->N, Co, p.Ho, p.Wo, p.S, p.Wl, p.Sh, p.Hlo, btmp, st, gp, psg,
                                          nullptr);
        else
            s = launch_prep_pieces(gy, gp, (long long)ng, psg, st);
        if (s) return s;
        const long long blocks = (long long)d->N * d->H * ((d->W + 31) / 32);
        if (blocks > 0x7fffffffLL) return HC_ERR_UNSUPPORTED;
        prep_pieces_nhwc_kernel<<<(unsigned)blocks, 256, 0, st>>>(x, xp, Ci, d->H, d->W);
        if ((s = launched("prep_pieces_nhwc_kernel", st))) return s;
        TcParams tp{};
        tp.mode = 1;
        tp.fmt = 1;
        tp.bmn = 1;
        tp.Co = Co;
        tp.Ci = Ci;
        tp.S = p.Q;
        tp.Sw = p.S;
        tp.own_h = p.Hlo;
        tp.J = tc_wgrad_splits(d, p);
        tp.own_w = p.Wl;
        tp.row_chunks = p.Wl / BKH;
        tp.Ho = p.Ho;
        tp.kh = K;
        tp.kw = K;
        tp.pad = d->padding;
        tp.taps = KK;
        tp.mblocks = Co / BM;
        tp.nblocks = Ci / WG_SLOT;
        tp.slots = KK * tp.nblocks;
        tp.kvalid = Ci;
        tp.shard_chunks = (long long)d->N * p.Hlo * tp.row_chunks;
        tp.units = tp.mblocks * ((tp.slots + 1) / 2) * tp.J * p.Q;
        tp.part = part;
        tp.N = d->N;
        CUtensorMap ma, mb;
        if ((s = pieces_rows_map(&ma, gp, d->N, Co, p.Ho, p.Wo, BM, psg)) ||
            (s = pieces_nhwc_map(&mb, xp, d->N, Ci, d->H, d->W)))
            return s;
        if ((s = launch_conv_pass(WG_BN, ma, mb, tp, st))) return s;
        wgrad_reduce_kernel<<<(unsigned)(p.Q * Co), 256, 0, st>>>(part, gwp, tp.J, KK, Co, Ci);
        if ((s = launched("wgrad_reduce_kernel", st))) return s;
    }
    return HC_OK;
}

// ---------------------------------------------------------------------------
// Convolutions on bf16 pieces: 1x1 (stride 1, no padding) and k = stride = s
// (no padding) as a 1x1 conv of the space-to-depth image.  The pieces keep
// NCHW order -- of x, or of the space-to-depth image [N][s*s*C][Ho][Wo] --
// and of grad_output.  A 1x1 conv pass treats the H*W pixels of an image as
// one flat row (Ho = 1, Wo = H*W); a space-to-depth pass tiles output rows and
// stores grad_input depth-to-space.  K past the last channel reads as zeros
// (TMA fill), so no padded copies are written.  The weight gradient walks a
// shard's own columns as in the tf32 pass.
namespace {
struct Bf16View {
    bool s2d;
    int s, K;     // stride; GEMM depth of the forward pass (C_in, or s*s*C_in)
    long long P;  // pixels of one output image
};
Bf16View bf16_view(const hc_conv_desc* d, const Plan& p) {
    Bf16View v;
    v.s2d = is_s2d(d);
    v.s = d->stride;
    v.K = v.s2d ? v.s * v.s * d->C_in : d->C_in;
    v.P = (long long)p.Ho * p.Wo;
    return v;
}
}  // namespace

bool bf16_supported(const hc_conv_desc* d, const Plan& p) {
    if (d->C_out % BM) return false;  // M blocks of the forward pass
    const Bf16View v = bf16_view(d, p);
    if (v.s2d) {
        // row tiles of 128 / 256 output columns; 4*s input columns per prep item
        if (v.s > 4 || d->H % v.s || d->W % v.s || p.Ho != d->H / v.s || p.Wo != d->W / v.s) return false;
        if (!pick_bn(p.Wo) || v.K % 8) return false;
    } else {
        if (d->groups != 1 || d->kh != 1 || d->kw != 1 || d->stride != 1 || d->padding != 0) return false;
        if (d->C_in % BM || v.P % 128) return false;  // grad_input M blocks; flat tiles of 128 / 256 pixels
    }
    // weight-gradient chunks of 32 pixels inside a shard's columns; 16-byte rows
    if ((p.Wl / v.s) % BKH || p.Wo % 8) return false;
    return (long long)d->N * v.K * v.P < (1LL << 36) && (long long)d->N * d->C_out * v.P < (1LL << 36);
}

// Workspace: forward  [x pieces][w pieces]
//            backward [gy pieces][w^T pieces][split-K partials][x pieces]; pass 2
//            (x's pieces taken from the forward workspace) stops before x pieces
size_t bf16_ws_bytes(const hc_conv_desc* d, const Plan& p, int pass) {
    const Bf16View v = bf16_view(d, p);
    const size_t psx = piece_stride((long long)d->N * v.K * v.P), psg = piece_stride((long long)d->N * d->C_out * v.P);
    const size_t psw = piece_stride((long long)d->C_out * v.K);
    if (pass == 0) return al256(6 * psx) + al256(6 * psw);
    const int Kp = v.s2d ? s2d_kp(d) : d->C_in;  // partial row pitch: whole 128-column slots
    const size_t part = al256(4 * (size_t)p.Q * tc_wgrad_splits(d, p) * d->C_out * Kp);
    return al256(6 * psg) + al256(6 * psw) + part + (pass == 2 ? 0 : al256(6 * psx));
}

static hc_status prep_x_pieces(const hc_conv_desc* d, const Plan& p, const Bf16View& v, const float* x, void* out,
                               long long ps, cudaStream_t st) {
    if (!v.s2d) return launch_prep_pieces(x, out, (long long)d->N * d->C_in * v.P, ps, st);
    const long long items = (long long)d->N * d->C_in * d->H * (p.Wo / 4);
    long long blocks = (items + 255) / 256;
    if (blocks > 152LL * 32) blocks = 152LL * 32;
    if (blocks < 1) blocks = 1;
    uint2* o = reinterpret_cast<uint2*>(out);
    if (v.s == 2)
        prep_s2d_pieces_kernel<2><<<(unsigned)blocks, 256, 0, st>>>(x, o, d->C_in, d->H, d->W, items, ps / 4);
    else if (v.s == 3)
        prep_s2d_pieces_kernel<3><<<(unsigned)blocks, 256, 0, st>>>(x, o, d->C_in, d->H, d->W, items, ps / 4);
    else if (v.s == 4)
        prep_s2d_pieces_kernel<4><<<(unsigned)blocks, 256, 0, st>>>(x, o, d->C_in, d->H, d->W, items, ps / 4);
    else
        return HC_ERR_UNSUPPORTED;
    return launched("prep_s2d_pieces_kernel", st);
}

// Output stores of a bf16 conv pass: a short K (under 16 chunks) leaves the
// 128 KB output tile of a unit a large share of the copy traffic, and the TMA
// store boxes win; a long K gains more from the third ring stage that plain
// per-thread stores leave room for (measured on the block's 1x1 and stem convs).
static const CUtensorMap* bf16_store_map(const TcParams& tp, const CUtensorMap* my) {
    return tp.chunks < 16 ? my : nullptr;
}

// The conv-pass tiling: flat rows of BN pixels (1x1) or BN-column segments of
// output rows (space-to-depth).
static void bf16_tiles(const Plan& p, const Bf16View& v, TcParams& tp, int* BN) {
    if (v.s2d) {
        *BN = pick_bn(p.Wo);
        tp.Ho = p.Ho;
        tp.Wo = p.Wo;
    } else {
        *BN = v.P % 256 == 0 ? 256 : 128;
        tp.Ho = 1;
        tp.Wo = (int)v.P;
    }
    tp.tiles_w = tp.Wo / *BN;
}

hc_status launch_bf16_fwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* b,
                          float* y, void* ws, cudaStream_t st, bool gelu_in) {
    const Bf16View v = bf16_view(d, p);
    if (gelu_in && v.s2d) return HC_ERR_UNSUPPORTED;
    const int Co = d->C_out;
    const long long wsz = (long long)Co * v.K;
    const long long psx = piece_stride((long long)d->N * v.K * v.P), psw = piece_stride(wsz);
    char* q = (char*)ws;
    void* xp = q;
    q += al256(6 * psx);
    void* ap = q;
    hc_status e;
    if ((e = gelu_in ? launch_prep_pieces(x, xp, (long long)d->N * d->C_in * v.P, psx, st, true)
                     : prep_x_pieces(d, p, v, x, xp, psx, st)))
        return e;
    if (v.s2d) {
        prep_weight_s2d_pieces_kernel<<<cdiv(wsz, 256), 256, 0, st>>>(w, (__nv_bfloat16*)ap, Co, d->C_in, v.s, 0,
                                                                      psw);
        e = launched("prep_weight_s2d_pieces_kernel", st);
    } else {
        e = launch_prep_pieces(w, ap, wsz, psw, st);
    }
    if (e) return e;
    TcParams tp{};
    int BN;
    bf16_tiles(p, v, tp, &BN);
    tp.mode = 0;
    tp.fmt = 1;
    tp.N = d->N;
    tp.M = Co;
    tp.Kc = v.K;
    tp.kh = 1;
    tp.kw = 1;
    tp.pad = 0;
    tp.mblocks = Co / BM;
    tp.chunks = (v.K + BKH - 1) / BKH;
    tp.units = tp.mblocks * d->N * tp.Ho * tp.tiles_w;
    tp.bias = b;
    tp.out = y;
    CUtensorMap ma, mb, my;
    if ((e = pieces_weight_map(&ma, ap, Co, v.K, psw)) || (e = pieces_mn_map(&mb, xp, d->N, v.K, v.P, BN, psx)) ||
        (e = out_map(&my, y, d->N, Co, tp.Ho, tp.Wo)))
        return e;
    return launch_conv_pass(BN, ma, mb, tp, st, bf16_store_map(tp, &my));
}

hc_status launch_bf16_bwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* gy,
                          float* gx, float* gwp, bool want_w, void* ws, const void* fwd_ws, float* gbp,
                          float* btmp, cudaStream_t st, bool gelu_in, const float* gelu_y) {
    const Bf16View v = bf16_view(d, p);
    if ((gelu_in || gelu_y) && v.s2d) return HC_ERR_UNSUPPORTED;
    const int Co = d->C_out;
    const long long wsz = (long long)Co * v.K;
    const long long psx = piece_stride((long long)d->N * v.K * v.P);
    const long long psg = piece_stride((long long)d->N * Co * v.P), psw = piece_stride(wsz);
    const int Kp = v.s2d ? s2d_kp(d) : d->C_in;  // partial row pitch: whole 128-column slots
    char* q = (char*)ws;
    void* gp = q;
    q += al256(6 * psg);
    void* ap = q;
    q += al256(6 * psw);
    float* part = (float*)q;
    q += al256(4 * (size_t)p.Q * tc_wgrad_splits(d, p) * Co * Kp);
    // x's pieces: from the forward workspace (its first region) or built here
    void* xp = fwd_ws ? const_cast<void*>(fwd_ws) : (void*)q;
    hc_status e;
    // grad_output's pieces serve both passes; the bias-gradient partials, when
    // asked for, are summed in the same read of grad_output.  With gelu_y the
    // output gradient is gy * GELU'(gelu_y), formed as gy is read.
    if (gbp)
        e = launch_bias_grad_partials(gy, gbp, d->N, Co, p.Ho, p.Wo, p.S, p.Wl / v.s, p.Sh, p.Hlo, btmp, st, gp,
                                      psg, gelu_y);
    else
        e = launch_prep_pieces(gy, gp, (long long)d->N * Co * v.P, psg, st, false, gelu_y);
    if (e) return e;
    if (gx) {  // D[m][px] = sum_co w^T[m][co] gy[co][px], m = ci (1x1) or (u*C + c)*s + v (depth-to-space)
        if (v.s2d)
            prep_weight_s2d_pieces_kernel<<<cdiv(wsz, 256), 256, 0, st>>>(w, (__nv_bfloat16*)ap, Co, d->C_in, v.s,
                                                                          1, psw);
        else
            prep_pieces_t_kernel<<<cdiv(wsz, 256), 256, 0, st>>>(w, (__nv_bfloat16*)ap, Co, d->C_in, psw);
        if ((e = launched("prep_pieces_t_kernel", st))) return e;
        TcParams tp{};
        int BN;
        bf16_tiles(p, v, tp, &BN);
        tp.mode = 0;
        tp.fmt = 1;
        tp.N = d->N;
        tp.M = v.K;
        tp.Kc = Co;
        tp.kh = 1;
        tp.kw = 1;
        tp.pad = 0;
        tp.mblocks = (v.K + BM - 1) / BM;
        tp.chunks = Co / BKH;
        tp.units = tp.mblocks * d->N * tp.Ho * tp.tiles_w;
        tp.bias = nullptr;
        tp.out = gx;
        CUtensorMap ma, mb, my;
        if ((e = pieces_weight_map(&ma, ap, v.K, Co, psw)) || (e = pieces_mn_map(&mb, gp, d->N, Co, v.P, BN, psg)))
            return e;
        if (v.s2d) {
            tp.d2s = v.s;
            tp.d2s_c = d->C_in;
            if ((e = launch_conv_pass(BN, ma, mb, tp, st))) return e;
        } else {
            if ((e = out_map(&my, gx, d->N, v.K, 1, (int)v.P))) return e;
            if ((e = launch_conv_pass(BN, ma, mb, tp, st, bf16_store_map(tp, &my)))) return e;
        }
    }
    if (want_w) {  // G[co][k] = sum over a shard's pixels of gy[co][px] x'[k][px]
        if (!fwd_ws && (e = gelu_in ? launch_prep_pieces(x, xp, (long long)d->N * d->C_in * v.P, psx, st, true)
                                    : prep_x_pieces(d, p, v, x, xp, psx, st)))
            return e;
        TcParams tp{};
        tp.mode = 1;
        tp.fmt = 1;
        tp.Co = Co;
        tp.Ci = Kp;
        tp.S = p.Q;
        tp.Sw = p.S;
        tp.own_h = p.Hlo;
        tp.J = tc_wgrad_splits(d, p);
        tp.own_w = p.Wl / v.s;
        tp.row_chunks = tp.own_w / BKH;
        tp.Ho = p.Ho;
        tp.kh = 1;
        tp.kw = 1;
        tp.pad = 0;
        tp.taps = 1;
        tp.mblocks = Co / BM;
        tp.nblocks = Kp / WG_SLOT;
        tp.slots = tp.nblocks;
        tp.kvalid = v.K;
        tp.shard_chunks = (long long)d->N * p.Hlo * tp.row_chunks;
        tp.units = tp.mblocks * ((tp.slots + 1) / 2) * tp.J * p.Q;
        tp.part = part;
        tp.N = d->N;
        CUtensorMap ma, mb;
        if ((e = pieces_rows_map(&ma, gp, d->N, Co, p.Ho, p.Wo, BM, psg)) ||
            (e = pieces_rows_map(&mb, xp, d->N, v.K, p.Ho, p.Wo, WG_BN, psx)))
            return e;
        if ((e = launch_conv_pass(WG_BN, ma, mb, tp, st))) return e;
        if (v.s2d)
            wgrad_reduce_s2d_kernel<<<(unsigned)(p.Q * Co), 256, 0, st>>>(part, gwp, tp.J, Co, d->C_in, v.s, Kp);
        else
            wgrad_reduce_kernel<<<(unsigned)(p.Q * Co), 256, 0, st>>>(part, gwp, tp.J, 1, Co, d->C_in);
        if ((e = launched("wgrad_reduce_kernel", st))) return e;
    }
    return HC_OK;
}

namespace {
// Self-test of the timeout path: wait on an mbarrier that nothing arrives on,
// for at most wait_ns of the global timer, then record HC_ERR_TIMEOUT exactly
// as a pipeline kernel that gave up would, and return.
__global__ void selftest_timeout_kernel(long long wait_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t0));
    while (!mbar_try(&bar, 0)) {
        asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
        if ((long long)(t - t0) > wait_ns) {
            atomicCAS(&g_tc_status, 0, (int)HC_ERR_TIMEOUT);
            return;
        }
    }
}
}  // namespace

hc_status launch_selftest_timeout(int wait_us, cudaStream_t st) {
    if (wait_us < 1 || wait_us > 2000000) return HC_ERR_INVALID_ARG;
    selftest_timeout_kernel<<<1, 32, 0, st>>>((long long)wait_us * 1000);
    return launched("selftest_timeout_kernel", st);
}

hc_status tc_take_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return HC_ERR_CUDA;
    }
    if (v) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int));
    }
    return (hc_status)v;
}

}  // namespace hc
