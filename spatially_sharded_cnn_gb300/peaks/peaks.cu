// peaks.cu -- microbenchmarks of the GB300 units the convolution kernels are
// bound by: the FP32 FMA pipe (scalar and packed FMA loops, FMAs with three
// distinct register operands), the 7x7 depthwise stencil and weight-gradient
// correlation with their tiles already in shared memory (the compute ceiling
// of those kernels), and the tcgen05 tensor pipe (kind::tf32 and kind::f16
// MMA loops from shared memory into tensor memory).  A measurement aid for the
// roofline denominators; not part of the convolution library.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr int K = 7, P = 3;
constexpr long long kWait = 4000000000LL;  // clock cycles, about 2 s

// ---------------- FP32 FMA loops ----------------------------------------------
// kind 0: acc = acc * a + b (two loop-invariant operands); 1: the same as packed
// pairs (fma.rn.f32x2); 2: acc[i] += w[k] * x[(i + k) % 8], three distinct registers.
template <int KIND>
__global__ void __launch_bounds__(256) fma_loop(float* out, const float* src, int iters) {
    float acc[16], w[8], x[8];
#pragma unroll
    for (int i = 0; i < 16; i++) acc[i] = threadIdx.x * 1e-3f + i;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        w[i] = src[i];
        x[i] = src[8 + i] + threadIdx.x;
    }
    const float a = src[16], b = src[17];
    for (int it = 0; it < iters; it++) {
        if (KIND == 0) {
#pragma unroll
            for (int u = 0; u < 8; u++)
#pragma unroll
                for (int i = 0; i < 16; i++) acc[i] = fmaf(acc[i], a, b);
        } else if (KIND == 1) {
            const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
#pragma unroll
            for (int u = 0; u < 8; u++)
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const float2 r = __ffma2_rn(make_float2(acc[i], acc[i + 1]), a2, b2);
                    acc[i] = r.x;
                    acc[i + 1] = r.y;
                }
        } else {
#pragma unroll
            for (int k = 0; k < 8; k++)
#pragma unroll
                for (int i = 0; i < 16; i++) acc[i] = fmaf(w[k], x[(i + k) & 7], acc[i]);
        }
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; i++) s += acc[i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// ---------------- the depthwise stencil, compute only --------------------------
// The convolution kernels' register blocking: each thread an 8-row x 4-column
// output block, per input row three 16-byte shared loads and up to 7 * 4 * 7
// FMAs with the 49 weights in registers.  Every job reads another of NST
// shared-memory stages (filled once), so no work is loop-invariant.
constexpr int SMW = 136;
constexpr int ST_WARPS = 8, ST_CTAS = 2, ST_NST = 2, ST_R = 8 * ST_WARPS + 2 * P;

__global__ void __launch_bounds__(ST_WARPS * 32, ST_CTAS)
    stencil_ceiling(const float* __restrict__ w, float* __restrict__ out, int jobs) {
    extern __shared__ __align__(16) float sm[];
    for (int i = threadIdx.x; i < ST_NST * ST_R * SMW; i += blockDim.x)
        sm[i] = (float)((i * 2654435761u) >> 20) * 1e-6f - 0.5f;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float wt[K][K];
    for (int u = 0; u < K; u++)
        for (int v = 0; v < K; v++) wt[u][v] = __ldg(w + (blockIdx.x & 127) * 49 + u * K + v);
    float* op = out + (size_t)(blockIdx.x * ST_WARPS + warp) * 8 * 128;
    for (int q = 0; q < jobs; q++) {
        const float* s = sm + (q % ST_NST) * ST_R * SMW;
        float acc[8][4];
#pragma unroll
        for (int r = 0; r < 8; r++)
#pragma unroll
            for (int j = 0; j < 4; j++) acc[r][j] = 0.0f;
#pragma unroll
        for (int i = 0; i < 8 + 2 * P; i++) {
            const float4* rp = reinterpret_cast<const float4*>(s + (warp * 8 + i) * SMW + 4 * lane);
            const float4 a = rp[0], b = rp[1], c = rp[2];
            const float xs[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
#pragma unroll
            for (int r = 0; r < 8; r++) {
                const int u = i - r;
                if (u >= 0 && u < K) {
#pragma unroll
                    for (int v = 0; v < K; v++)
#pragma unroll
                        for (int jj = 0; jj < 4; jj++) acc[r][jj] = fmaf(wt[u][v], xs[jj + v + 1], acc[r][jj]);
                }
            }
        }
        float* o = op + (size_t)(q & 7) * (gridDim.x * ST_WARPS * 8 * 128);
#pragma unroll
        for (int r = 0; r < 8; r++)
            *reinterpret_cast<float4*>(o + r * 128 + 4 * lane) = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    }
}

// The weight-gradient correlation of the backward pass: each thread the 49
// accumulators gw[u][v] += g[r][c] * x[r + u][c + v] over 4-row x 4-column
// blocks of grad_output, x rows from shared memory.
constexpr int CR_WARPS = 8, CR_NST = 3, CR_R = 8 * CR_WARPS + 2 * P;

__global__ void __launch_bounds__(CR_WARPS * 32, 1) correlation_ceiling(float* __restrict__ out, int jobs) {
    extern __shared__ __align__(16) float sm[];
    for (int i = threadIdx.x; i < 2 * CR_NST * CR_R * SMW; i += blockDim.x)
        sm[i] = (float)((i * 2654435761u) >> 20) * 1e-6f - 0.5f;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float gw[K][K];
#pragma unroll
    for (int u = 0; u < K; u++)
#pragma unroll
        for (int v = 0; v < K; v++) gw[u][v] = 0.0f;
    for (int q = 0; q < jobs; q++) {
        const float* gys = sm + (q % CR_NST) * 2 * CR_R * SMW;
        const float* xs = gys + CR_R * SMW;
#pragma unroll 1
        for (int h = 0; h < 2; h++) {
            const int row0 = warp * 8 + 4 * h;
            float g[4][4];
#pragma unroll
            for (int r = 0; r < 4; r++) {
                const float4 v4 = *reinterpret_cast<const float4*>(gys + (P + row0 + r) * SMW + 4 + 4 * lane);
                g[r][0] = v4.x;
                g[r][1] = v4.y;
                g[r][2] = v4.z;
                g[r][3] = v4.w;
            }
#pragma unroll
            for (int i = 0; i < 4 + 2 * P; i++) {
                const float4* rp = reinterpret_cast<const float4*>(xs + (row0 + i) * SMW + 4 * lane);
                const float4 a = rp[0], b = rp[1], c = rp[2];
                const float xr[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
#pragma unroll
                for (int r = 0; r < 4; r++) {
                    const int u = i - r;
                    if (u >= 0 && u < K) {
#pragma unroll
                        for (int jj = 0; jj < 4; jj++)
#pragma unroll
                            for (int v = 0; v < K; v++) gw[u][v] = fmaf(g[r][jj], xr[jj + v + 1], gw[u][v]);
                    }
                }
            }
        }
    }
    float t = 0.0f;
#pragma unroll
    for (int u = 0; u < K; u++)
#pragma unroll
        for (int v = 0; v < K; v++) t += gw[u][v] * (1 + u + v);
    out[blockIdx.x * blockDim.x + threadIdx.x] = t;
}

// ---------------- tcgen05 MMA loop ------------------------------------------------
__device__ __forceinline__ unsigned su32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

// Shared-memory matrix descriptor, 128-byte swizzle, K-major (SBO = 8-row group stride).
__device__ __forceinline__ uint64_t sdesc_sw128(const void* p, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((su32(p) >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;  // leading byte offset (unused for swizzled K-major tiles)
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// Instruction descriptors: D fp32; A, B tf32 (kind::tf32) or bf16 (kind::f16); K-major; N, M.
__host__ __device__ constexpr uint32_t idesc(int kind, int M, int N) {
    return (1u << 4) | ((kind ? 1u : 2u) << 7) | ((kind ? 1u : 2u) << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

constexpr int MMA_M = 128;

// One thread per CTA issues `iters` MMAs (M = 128, N = MMA_N, K = 8 tf32 or 16
// bf16: one 32-byte k-step of 128-byte swizzled operand rows, cycling over the
// four k-steps of the tiles) accumulating into one TMEM tile, commits them to an
// mbarrier, and the CTA waits for it (bounded) before freeing the tensor memory.
// Operand values do not matter for the rate; the tiles are zero.
template <int KIND, int MMA_N>
__global__ void __launch_bounds__(128) mma_loop(int iters, int* status) {
    constexpr uint32_t TCOLS = MMA_N < 32 ? 32 : MMA_N;
    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char* base = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    unsigned char* a = base;                       // 128 rows x 128 bytes
    unsigned char* b = base + MMA_M * 128;         // MMA_N rows x 128 bytes
    uint64_t* bar = (uint64_t*)(b + MMA_N * 128);
    uint32_t* slot = (uint32_t*)(bar + 1);
    for (int i = threadIdx.x; i < (MMA_M + MMA_N) * 128 / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(base)[i] = make_uint4(0, 0, 0, 0);
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(su32(slot)),
                     "r"(TCOLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    const uint32_t tmem = *slot;
    if (threadIdx.x == 0) {
        const uint32_t id = idesc(KIND, MMA_M, MMA_N);
        for (int it = 0; it < iters; it++) {
            const int ks = it & 3;
            const uint64_t ad = sdesc_sw128(a + 32 * ks, 1024), bd = sdesc_sw128(b + 32 * ks, 1024);
            const uint32_t acc = it > 0;
            if (KIND)
                asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                             " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
                             "l"(ad), "l"(bd), "r"(id), "r"(acc)
                             : "memory");
            else
                asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                             " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
                             "l"(ad), "l"(bd), "r"(id), "r"(acc)
                             : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(su32(bar))
                     : "memory");
    }
    // every thread waits (bounded) for the committed MMAs
    const long long t0 = clock64();
    bool ok = true;
    for (;;) {
        unsigned done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(su32(bar))
            : "memory");
        if (done) break;
        if (clock64() - t0 > kWait) {
            ok = false;
            break;
        }
    }
    if (!ok && threadIdx.x == 0) atomicExch(status, 1);
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(TCOLS) : "memory");
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

}  // namespace

extern "C" {

// Floats the `out` buffer of the FP32 loops and ceilings needs.
long long hcp_out_floats(void) { return (long long)sm_count() * 8 * 8 * ST_WARPS * 8 * 128 + 4096; }

// kind 0 / 1 / 2: FMA loop with two loop-invariant operands / packed pairs /
// three distinct registers; `ctas_per_sm` 256-thread CTAs per SM.  src: 18
// floats.  *flops: the FP32 FLOPs the launch does (2 per FMA).
int hcp_fp32_loop(int kind, int iters, int ctas_per_sm, float* out, const float* src, void* stream, double* flops) {
    const int grid = sm_count() * ctas_per_sm;
    cudaStream_t st = (cudaStream_t)stream;
    if (kind == 0)
        fma_loop<0><<<grid, 256, 0, st>>>(out, src, iters);
    else if (kind == 1)
        fma_loop<1><<<grid, 256, 0, st>>>(out, src, iters);
    else
        fma_loop<2><<<grid, 256, 0, st>>>(out, src, iters);
    *flops = 2.0 * 16 * 8 * (double)iters * grid * 256;
    return (int)cudaGetLastError();
}

// kind 0: the depthwise 7x7 stencil (two 8-warp CTAs per SM); kind 1: the
// weight-gradient correlation (one 8-warp CTA per SM); `jobs` 64-row x
// 128-column tiles per CTA.  w: 128 * 49 floats.
int hcp_stencil(int kind, int jobs, const float* w, float* out, void* stream, double* flops) {
    cudaStream_t st = (cudaStream_t)stream;
    const int sms = sm_count();
    if (kind == 0) {
        const int smem = ST_NST * ST_R * SMW * 4;
        if (cudaFuncSetAttribute(stencil_ceiling, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) return -2;
        stencil_ceiling<<<sms * ST_CTAS, ST_WARPS * 32, smem, st>>>(w, out, jobs);
        *flops = 2.0 * 49 * (double)sms * ST_CTAS * ST_WARPS * 8 * 128 * jobs;
    } else {
        const int smem = 2 * CR_NST * CR_R * SMW * 4;
        if (cudaFuncSetAttribute(correlation_ceiling, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) return -2;
        correlation_ceiling<<<sms, CR_WARPS * 32, smem, st>>>(out, jobs);
        *flops = 2.0 * 49 * (double)sms * CR_WARPS * 8 * 128 * jobs;
    }
    return (int)cudaGetLastError();
}

// kind 0: tcgen05.mma kind::tf32 (M 128, N 256, K 8); kind 1: kind::f16 with
// bf16 operands (K 16); one CTA per SM, `iters` MMAs each.  kind 2: kind::tf32
// with N 16 (the narrowest M 128 shape), two CTAs per SM issuing side by side:
// the floor of the tensor pipe's time per MMA, which a narrow MMA cannot go
// below.  status: device int, set to 1 if a CTA gave up waiting for its MMAs.
// *flops: the FLOPs the MMAs issued (2 M N K each).
int hcp_mma(int kind, int iters, int* status, void* stream, double* flops) {
    cudaStream_t st = (cudaStream_t)stream;
    const int sms = sm_count();
    const int N = kind == 2 ? 16 : 256, ctas = kind == 2 ? 2 * sms : sms;
    const int smem = (MMA_M + N) * 128 + 1024 + 64;
    const auto A = cudaFuncAttributeMaxDynamicSharedMemorySize;
    if (kind == 0) {
        if (cudaFuncSetAttribute(mma_loop<0, 256>, A, smem)) return -2;
        mma_loop<0, 256><<<ctas, 128, smem, st>>>(iters, status);
    } else if (kind == 1) {
        if (cudaFuncSetAttribute(mma_loop<1, 256>, A, smem)) return -2;
        mma_loop<1, 256><<<ctas, 128, smem, st>>>(iters, status);
    } else {
        if (cudaFuncSetAttribute(mma_loop<0, 16>, A, smem)) return -2;
        mma_loop<0, 16><<<ctas, 128, smem, st>>>(iters, status);
    }
    *flops = 2.0 * MMA_M * N * (kind == 1 ? 16 : 8) * (double)iters * ctas;
    return (int)cudaGetLastError();
}

}  // extern "C"
