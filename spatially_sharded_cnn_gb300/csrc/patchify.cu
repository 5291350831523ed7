// patchify.cu -- weight and bias gradient of the ConvNeXt "patchify" stem
// (4x4 kernel, stride 4, no padding, 3 input channels) as a direct FP32
// reduction:
//
//   gw[co][ci][kh][kw] = sum over (n, ho, wo) of gy[n][co][ho][wo] * x[n][ci][4 ho + kh][4 wo + kw]
//   gb[co]             = sum over (n, ho, wo) of gy[n][co][ho][wo]
//
// taken per grid shard over that shard's own output rows and columns (the
// per-device _Partial gradients of the NVIDIA blog "Perception model training
// for autonomous vehicles with tensor parallelism", design section; kwkr.cn
// news/18980 section 2.2) and summed in shard order.  With stride = kernel the
// shards' input blocks do not overlap, so there is no halo.
//
// Why not the tensor cores: the contraction (over N * Ho * Wo pixels) has only
// 48 output columns per channel, and fp32 accuracy on them needs grad_output
// split into pieces first -- two to three ALU instructions per value of the
// largest tensor, about as much issue time as the FP32 reduction itself, plus
// the pieces' HBM traffic.  The reduction reads x and grad_output once.
//
// Layout of the work: CTA b serves one (grid shard, 256-channel block) group and
// a contiguous range of its jobs; a job is one output row segment of 32 pixels
// (n, ho, wo0 .. wo0 + 31), fed by two TMA boxes into a 4-stage mbarrier ring:
// grad_output [256 co][32 px] (128-byte swizzle) and the image rows under it
// [3 ci][4 kh][128 columns].  Warp w handles kernel row kh = w % 4 and pixel
// half w / 4 of every job; lane l holds channels co = 32 j + l (j < 8) and sums
// 8 x 3 x 4 weight terms (ci, kw) in registers (plus two channels' bias terms),
// so every grad_output value it loads feeds 12 FMAs and every image value (a
// warp-wide broadcast) 8.  At the end the two pixel halves are added (half 0 +
// half 1) and the CTA's partial goes to its slot; the shard-partials reduction
// then sums the slots in order.  Every wait is bounded; a CTA that times out
// records HC_ERR_TIMEOUT and drains its copies before it exits.
#include "common.cuh"

namespace hc {
namespace {

constexpr int PW_CO = 256;                    // output channels per CTA group
constexpr int PW_PX = 32;                     // output pixels per job
constexpr int PW_CI = 3, PW_K = 4;            // input channels, kernel = stride
constexpr int PW_KW = PW_CI * PW_K * PW_K;    // 48 weights per output channel
constexpr int PW_SLOT = PW_KW + 1;            // + the bias
constexpr int PW_NST = 4;                     // ring stages
constexpr int PW_WARPS = 8;
constexpr unsigned PW_GY = PW_CO * PW_PX * 4;                  // 32 KB
constexpr unsigned PW_X = PW_CI * PW_K * PW_PX * PW_K * 4;     // 6 KB
constexpr unsigned PW_STAGE = PW_GY + PW_X;                    // 38 KB, a multiple of 1024
constexpr int PW_RED = 4 * 32 * (PW_CI * PW_K * 8 + 2);        // floats: pixel half 1's sums
constexpr long long kWaitCycles = 4000000000LL;                // about 2 s
static_assert(PW_STAGE % 1024 == 0, "stages keep the 128-byte swizzle's 1024-byte alignment");
static_assert(PW_RED * 4 <= (int)(PW_NST * PW_STAGE), "the flush reuses the ring");

__device__ int g_pw_status;

__device__ __forceinline__ unsigned su32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* b, unsigned n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(su32(b)), "r"(n) : "memory");
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
__device__ __forceinline__ bool mbar_wait(uint64_t* b, unsigned parity) {
    if (mbar_try(b, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try(b, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}
__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* m, int c0, int c1, int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n" ::
            "r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(su32(bar))
        : "memory");
}

struct PwArgs {
    int N, Co, Hlo, Wlo;  // images, output channels, owned output rows / columns per grid shard
    int S;                // column shards (grid shard q = row block * S + column block)
    int G;                // CTAs per (grid shard, channel block) group
    float* tile_part;     // [Q][Co][G][PW_SLOT]
};

__global__ void __launch_bounds__(PW_WARPS * 32, 1)
    patchify_wgrad_kernel(const __grid_constant__ CUtensorMap gymap, const __grid_constant__ CUtensorMap xmap,
                          PwArgs a) {
    extern __shared__ unsigned char pw_smem[];
    unsigned char* ring = (unsigned char*)(((uintptr_t)pw_smem + 1023) & ~(uintptr_t)1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + PW_NST * PW_STAGE);
    int* done = reinterpret_cast<int*>(full + PW_NST);  // [PW_NST] warps finished with the stage
    int* issued = done + PW_NST;                        // jobs whose copies have been issued
    int* failed = issued + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kh = warp & 3, half = warp >> 2;

    const int grp = blockIdx.x / a.G, g = blockIdx.x - grp * a.G;
    const int cbs = a.Co / PW_CO, q = grp / cbs, cb = grp - q * cbs;
    const int rs = q / a.S, cs = q - rs * a.S;
    const int chunks = a.Wlo / PW_PX;
    const long long per = (long long)a.N * a.Hlo * chunks;
    const long long j0 = g * per / a.G;
    const int jobs = (int)((g + 1) * per / a.G - j0);

    // Job k's copies (chunk fastest, then output row, then image).  Any warp's
    // lane 0 may issue (the last one done with a stage), so the coordinates come
    // from k alone.
    auto issue = [&](int k) {
        const long long j = j0 + k, r = j / chunks;
        const int cch = (int)(j - r * chunks), chl = (int)(r % a.Hlo), cn = (int)(r / a.Hlo);
        uint64_t* bar = full + (k % PW_NST);
        unsigned char* st = ring + (k % PW_NST) * PW_STAGE;
        const int ho = rs * a.Hlo + chl, wo0 = cs * a.Wlo + cch * PW_PX;
        mbar_expect_tx(bar, PW_STAGE);
        tma_3d(st, &gymap, wo0, ho, cn * a.Co + cb * PW_CO, bar);
        tma_3d(st + PW_GY, &xmap, PW_K * wo0, PW_K * ho, cn * PW_CI, bar);
    };
    if (tid == 0) {
        for (int s = 0; s < PW_NST; s++) {
            mbar_init(full + s, 1);
            done[s] = 0;
        }
        *failed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        const int first = jobs < PW_NST ? jobs : PW_NST;
        for (int k = 0; k < first; k++) issue(k);
        *issued = first;
    }
    __syncthreads();

    float acc[8][PW_CI][PW_K];
    float gb0 = 0.0f, gb1 = 0.0f;  // bias terms of channels j = 2 kh and 2 kh + 1
#pragma unroll
    for (int j = 0; j < 8; j++)
#pragma unroll
        for (int ci = 0; ci < PW_CI; ci++)
#pragma unroll
            for (int kw = 0; kw < PW_K; kw++) acc[j][ci][kw] = 0.0f;

    int s = 0;
    unsigned ph = 0;
    for (int k = 0; k < jobs; k++) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(full + s, ph));
        if (!ok) {
            if (lane == 0) {
                atomicCAS(&g_pw_status, 0, (int)HC_ERR_TIMEOUT);
                *reinterpret_cast<volatile int*>(failed) = 1;
            }
            break;
        }
        const float* gys = reinterpret_cast<const float*>(ring + s * PW_STAGE);
        const float* xs = gys + PW_GY / 4;
#pragma unroll
        for (int p4 = 0; p4 < 4; p4++) {
            const int c4 = half * 4 + p4;  // 16-byte chunk of the 32-pixel row
            float4 gv[8];
#pragma unroll
            for (int j = 0; j < 8; j++)  // row co = 32 j + lane; the swizzle XORs the chunk with co % 8
                gv[j] = *reinterpret_cast<const float4*>(gys + (j * 32 + lane) * PW_PX + ((c4 ^ (lane & 7)) << 2));
#pragma unroll
            for (int j = 0; j < 8; j++)
                if ((j >> 1) == kh) {
                    const float t = (gv[j].x + gv[j].y) + (gv[j].z + gv[j].w);
                    if (j & 1)
                        gb1 += t;
                    else
                        gb0 += t;
                }
            // the image values of the 4 pixels: per channel, pixel p's four kw columns
            float4 xv[PW_CI][4];
#pragma unroll
            for (int ci = 0; ci < PW_CI; ci++)
#pragma unroll
                for (int p = 0; p < 4; p++)
                    xv[ci][p] = *reinterpret_cast<const float4*>(xs + (ci * PW_K + kh) * (PW_PX * PW_K) + c4 * 16 +
                                                                 4 * p);
            // acc[j][ci][kw] += gy[j][p] * x[ci][p][kw], kw in pairs (packed f32x2 FMAs: each
            // lane one fused multiply-add, the same sums in the same order as scalar FMAs)
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const float g4[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
#pragma unroll
                for (int p = 0; p < 4; p++) {
                    const float2 gg = make_float2(g4[p], g4[p]);
#pragma unroll
                    for (int ci = 0; ci < PW_CI; ci++) {
                        const float2 lo = __ffma2_rn(gg, make_float2(xv[ci][p].x, xv[ci][p].y),
                                                     make_float2(acc[j][ci][0], acc[j][ci][1]));
                        const float2 hi = __ffma2_rn(gg, make_float2(xv[ci][p].z, xv[ci][p].w),
                                                     make_float2(acc[j][ci][2], acc[j][ci][3]));
                        acc[j][ci][0] = lo.x;
                        acc[j][ci][1] = lo.y;
                        acc[j][ci][2] = hi.x;
                        acc[j][ci][3] = hi.y;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(done + s, 1) == PW_WARPS - 1) {  // the last warp out refills the stage
                done[s] = 0;
                __threadfence_block();
                if (k + PW_NST < jobs) {
                    issue(k + PW_NST);
                    atomicAdd(issued, 1);
                }
            }
        }
        if (++s == PW_NST) {
            s = 0;
            ph ^= 1u;
        }
    }
    __syncthreads();
    if (*failed) {  // wait (bounded) for the copies still in flight; no partial is written
        if (tid == 0) {
            const int last = *issued;
            for (int j = last - PW_NST > 0 ? last - PW_NST : 0; j < last; j++)
                mbar_wait(full + (j % PW_NST), (unsigned)((j / PW_NST) & 1));
        }
        return;
    }
    // pixel half 1 parks its sums in the (drained) ring; half 0 adds them to its own
    float* red = reinterpret_cast<float*>(ring) + (size_t)((warp & 3) * 32 + lane) * (PW_CI * PW_K * 8 + 2);
    if (half) {
#pragma unroll
        for (int j = 0; j < 8; j++)
#pragma unroll
            for (int ci = 0; ci < PW_CI; ci++)
#pragma unroll
                for (int kw = 0; kw < PW_K; kw++) red[(j * PW_CI + ci) * PW_K + kw] = acc[j][ci][kw];
        red[96] = gb0;
        red[97] = gb1;
    }
    __syncthreads();
    if (!half) {
        float* slot0 = a.tile_part + ((long long)q * a.Co + cb * PW_CO) * a.G * PW_SLOT + (long long)g * PW_SLOT;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            float* slot = slot0 + (long long)(j * 32 + lane) * a.G * PW_SLOT;
#pragma unroll
            for (int ci = 0; ci < PW_CI; ci++)
#pragma unroll
                for (int kw = 0; kw < PW_K; kw++)
                    slot[(ci * PW_K + kh) * PW_K + kw] = acc[j][ci][kw] + red[(j * PW_CI + ci) * PW_K + kw];
        }
        slot0[(long long)(2 * kh * 32 + lane) * a.G * PW_SLOT + PW_KW] = gb0 + red[96];
        slot0[(long long)((2 * kh + 1) * 32 + lane) * a.G * PW_SLOT + PW_KW] = gb1 + red[97];
    }
}

int pw_groups(const hc_conv_desc* d, const Plan& p) { return p.Q * (d->C_out / PW_CO); }
int pw_ctas_per_group(const hc_conv_desc* d, const Plan& p) {
    const int g = device_sm_count() / pw_groups(d, p);
    return g > 1 ? g : 1;
}

}  // namespace

bool patchify_wgrad_supported(const hc_conv_desc* d, const Plan& p) {
    return d->groups == 1 && d->C_in == PW_CI && d->kh == PW_K && d->kw == PW_K && d->stride == PW_K &&
           d->padding == 0 && d->C_out % PW_CO == 0 && d->W % PW_K == 0 && d->H % PW_K == 0 &&
           (p.Wl / PW_K) % PW_PX == 0 && p.Hlo > 0 && (long long)d->N * d->C_out < (1LL << 31) &&
           (long long)d->N * d->C_in < (1LL << 31);
}

size_t patchify_wgrad_ws_floats(const hc_conv_desc* d, const Plan& p) {
    return (size_t)p.Q * d->C_out * pw_ctas_per_group(d, p) * PW_SLOT;
}

hc_status launch_patchify_wgrad(const hc_conv_desc* d, const Plan& p, const float* x, const float* gy,
                                float* tile_part, float* gwp, float* gbp, float* gw, float* gb, cudaStream_t st) {
    const int Ho = p.Ho, Wo = p.Wo;
    CUtensorMap gm, xm;
    {
        const uint64_t dims[3] = {(uint64_t)Wo, (uint64_t)Ho, (uint64_t)d->N * d->C_out};
        const uint64_t strides[2] = {(uint64_t)Wo * 4, (uint64_t)Ho * Wo * 4};
        const uint32_t box[3] = {PW_PX, 1, PW_CO};
        hc_status s = make_tmap(&gm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, gy, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B);
        if (s) return s;
    }
    {
        const uint64_t dims[3] = {(uint64_t)d->W, (uint64_t)d->H, (uint64_t)d->N * d->C_in};
        const uint64_t strides[2] = {(uint64_t)d->W * 4, (uint64_t)d->H * d->W * 4};
        const uint32_t box[3] = {PW_PX * PW_K, PW_K, PW_CI};
        hc_status s = make_tmap(&xm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, x, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_NONE);
        if (s) return s;
    }
    const int G = pw_ctas_per_group(d, p), groups = pw_groups(d, p);
    const PwArgs a{d->N, d->C_out, p.Hlo, p.Wl / PW_K, p.S, G, tile_part};
    const size_t smem = 1024 + PW_NST * PW_STAGE + PW_NST * sizeof(uint64_t) + (PW_NST + 2) * sizeof(int);
    static std::atomic<unsigned long long> attr{0};
    once_per_device(attr, [&] {
        return cudaFuncSetAttribute(patchify_wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
               cudaSuccess;
    });
    patchify_wgrad_kernel<<<(unsigned)(groups * G), PW_WARPS * 32, smem, st>>>(gm, xm, a);
    hc_status s = launched("patchify_wgrad_kernel", st);
    if (s) return s;
    return launch_shard_partials(tile_part, gwp, gbp, gw, gb, p.Q, d->C_out, G, PW_KW, st);
}

hc_status pw_take_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_pw_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return HC_ERR_CUDA;
    }
    if (v) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_pw_status, &zero, sizeof(int));
    }
    return (hc_status)v;
}

}  // namespace hc
