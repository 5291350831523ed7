// reduce.cu -- fixed-order sums of partial results.
//
// The pages reduce the _Partial grad_weight / grad_bias of the shards with a
// cross-device reduce-sum (NVIDIA blog "Perception model training for
// autonomous vehicles with tensor parallelism", design section; kwkr.cn
// news/18980 section 2.2).  Here the shards' partials sit side by side in one
// buffer and are summed in shard order, so the result does not depend on
// timing and repeats bit for bit.
#include "common.cuh"

namespace hc {
namespace {

// out[k] = sum_{r = 0 .. rows-1} in[r * count + k], r ascending.  Consecutive
// threads take consecutive k, so every row is read coalesced.
__global__ void sum_rows_kernel(const float* __restrict__ in, float* __restrict__ out, int rows, long long count) {
    for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < count;
         k += (long long)gridDim.x * blockDim.x) {
        float acc = 0.0f;
        for (int r = 0; r < rows; r++) acc += __ldg(in + r * count + k);
        out[k] = acc;
    }
}

// Bias-gradient partial sums, stage 1: block (row shard a, slice, co) streams
// whole output rows (n, i), i among row shard a's rows, of its slice of
// grad_output channel co with 16-byte loads, 1024 columns at a time: each thread
// sums its four columns down the rows, then thread b adds the column sums of
// column shard b (shard of column j = j / own_w, the last shard taking the
// rest) in column order.  Every sum has a fixed order.
// part[(slice * Sh * S + a * S + b) * Co + co].  Needs Wo % 4 == 0, S <= 256,
// 256 threads.  PIECES: every float4 read also goes out as bf16 pieces
// (store_pieces4 at its own index), so one pass over grad_output serves both.
// GELU_D: the gradient read is gy * GELU'(hy) (hy: the pre-activation, gy's layout).
// Five resident blocks per SM (registers capped at 48): the GELU variant's erf / exp
// work then overlaps its loads best (measured 4, 5, 6, 8 blocks: 5 fastest).
template <bool PIECES, bool GELU_D>
__global__ void __launch_bounds__(256, 5) bias_rows_kernel(const float* __restrict__ gy, float* __restrict__ part, int N,
                                                        int Co, int Ho, int Wo, int S, int own_w, int Sh, int own_h,
                                                        int slices, uint2* __restrict__ pieces, long long ps4,
                                                        const float* __restrict__ hy) {
    __shared__ float cs[256];
    const int a = blockIdx.x / slices, slice = blockIdx.x - a * slices, co = blockIdx.y, tid = threadIdx.x;
    const int i0 = a * own_h, i1 = (a == Sh - 1) ? Ho : i0 + own_h, rows_a = i1 - i0;
    const int nrows = N * rows_a;
    const int r0 = (int)((long long)nrows * slice / slices), r1 = (int)((long long)nrows * (slice + 1) / slices);
    float total = 0.0f;  // thread b < S: column shard b's running sum
    for (int g0 = 0; g0 < Wo; g0 += 1024) {
        const int col = g0 + 4 * tid;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (col < Wo) {
            int row = r0;
            for (; row + 4 <= r1; row += 4) {  // four loads in flight, added in row order
                float4 v[4];
                long long e[4];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int n = (row + k) / rows_a, i = i0 + row + k - n * rows_a;
                    e[k] = (long long)co * Ho * Wo + col + ((long long)n * Co * Ho + i) * Wo;
                    v[k] = __ldg(reinterpret_cast<const float4*>(gy + e[k]));
                }
                if (GELU_D) {
                    float4 h[4];
#pragma unroll
                    for (int k = 0; k < 4; k++) h[k] = __ldg(reinterpret_cast<const float4*>(hy + e[k]));
#pragma unroll
                    for (int k = 0; k < 4; k++)
                        v[k] = make_float4(v[k].x * gelu_d(h[k].x), v[k].y * gelu_d(h[k].y), v[k].z * gelu_d(h[k].z),
                                           v[k].w * gelu_d(h[k].w));
                }
                if (PIECES) {
#pragma unroll
                    for (int k = 0; k < 4; k++) store_pieces4(v[k], pieces, e[k] / 4, ps4);
                }
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    acc.x += v[k].x;
                    acc.y += v[k].y;
                    acc.z += v[k].z;
                    acc.w += v[k].w;
                }
            }
            for (; row < r1; row++) {
                const int n = row / rows_a, i = i0 + row - n * rows_a;
                const long long e = (long long)co * Ho * Wo + col + ((long long)n * Co * Ho + i) * Wo;
                float4 v = __ldg(reinterpret_cast<const float4*>(gy + e));
                if (GELU_D) {
                    const float4 h = __ldg(reinterpret_cast<const float4*>(hy + e));
                    v = make_float4(v.x * gelu_d(h.x), v.y * gelu_d(h.y), v.z * gelu_d(h.z), v.w * gelu_d(h.w));
                }
                if (PIECES) store_pieces4(v, pieces, e / 4, ps4);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
        }
        cs[tid] = ((acc.x + acc.y) + acc.z) + acc.w;
        __syncthreads();
        if (tid < S) {
            const int j0 = tid * own_w, j1 = (tid == S - 1) ? Wo : j0 + own_w;
            const int lo = (j0 > g0 ? j0 : g0), hi = (j1 < g0 + 1024 ? j1 : g0 + 1024);
            for (int k = lo; k < hi; k += 4) total += cs[(k - g0) / 4];
        }
        __syncthreads();
    }
    if (tid < S) part[((long long)slice * Sh * S + (long long)a * S + tid) * Co + co] = total;
}

// Column sums, stage 1: tmp[g][k] = sum over rows r in group g (ascending) of
// in[r * stride + k].
__global__ void column_group_kernel(const float* __restrict__ in, float* __restrict__ tmp, int rows, int count,
                                    long long stride, int group) {
    const long long total = (long long)((rows + group - 1) / group) * count;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        const int k = (int)(q % count), g = (int)(q / count);
        const int r0 = g * group, r1 = r0 + group < rows ? r0 + group : rows;
        float s = 0.0f;
        for (int r = r0; r < r1; r++) s += __ldg(in + r * stride + k);
        tmp[q] = s;
    }
}

}  // namespace

size_t column_sum_tmp_floats(int rows, int count) {
    return (size_t)((rows + kColumnGroup - 1) / kColumnGroup) * count;
}

hc_status launch_column_sum(const float* in, float* out, int rows, int count, long long stride, float* tmp,
                            cudaStream_t st) {
    const long long total = (long long)((rows + kColumnGroup - 1) / kColumnGroup) * count;
    long long blocks = (total + 255) / 256;
    if (blocks > 152LL * 16) blocks = 152LL * 16;
    column_group_kernel<<<(unsigned)blocks, 256, 0, st>>>(in, tmp, rows, count, stride, kColumnGroup);
    hc_status s = launched("column_group_kernel", st);
    if (s) return s;
    return launch_sum_rows(tmp, out, (rows + kColumnGroup - 1) / kColumnGroup, count, st);
}

size_t bias_grad_ws_floats(int Co, int S) { return (size_t)kBiasSlices * S * Co; }

// Blocks of a bias row kernel variant resident on the whole GPU at once (one
// wave): 0 sums only, 1 with pieces, 2 with pieces of gy * GELU'(y).
static long long bias_wave(int variant) {
    static std::atomic<long long> caps[kMaxDevices][3];  // per device; host threads may call at once
    int dev = 0;
    cudaGetDevice(&dev);
    // an imposed SM count (hc_set_sm_count) is not cached
    const bool cached = dev >= 0 && dev < kMaxDevices && g_sm_override.load(std::memory_order_relaxed) == 0;
    long long v = cached ? caps[dev][variant].load(std::memory_order_relaxed) : 0;
    if (!v) {
        int sms = device_sm_count(), per = 0;
        if (variant == 2)
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, bias_rows_kernel<true, true>, 256, 0);
        else if (variant == 1)
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, bias_rows_kernel<true, false>, 256, 0);
        else
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, bias_rows_kernel<false, false>, 256, 0);
        cudaGetLastError();
        v = (long long)(sms > 0 ? sms : 1) * (per > 0 ? per : 1);
        if (cached) caps[dev][variant].store(v, std::memory_order_relaxed);
    }
    return v;
}

hc_status launch_bias_grad_partials(const float* gy, float* gbp, int N, int Co, int Ho, int Wo, int S, int own_w,
                                    int Sh, int own_h, float* tmp, cudaStream_t st, void* pieces, long long ps,
                                    const float* gelu_y) {
    if (Wo % 4 || own_w % 4 || S > 256 || Co > 65535 || Sh < 1 || (long long)N * Ho > 0x7fffffffLL || ps % 4 ||
        (gelu_y && !pieces))
        return HC_ERR_UNSUPPORTED;
    // about eight blocks per SM, at most kBiasSlices slices per row shard; then the
    // first slice count (upwards) whose last wave of resident blocks is >= 90 % full
    const long long rows_min = (long long)N * (Sh > 1 ? own_h : Ho);
    long long smax = rows_min < kBiasSlices ? rows_min : kBiasSlices;
    if (smax < 1) smax = 1;
    long long slices = (152LL * 8 + (long long)Co * Sh - 1) / ((long long)Co * Sh);
    if (slices > smax) slices = smax;
    if (slices < 1) slices = 1;
    const long long cap = bias_wave(gelu_y ? 2 : pieces ? 1 : 0);
    for (long long t = slices; t <= smax; t++) {
        const long long blocks = t * Sh * Co, waves = (blocks + cap - 1) / cap;
        if (blocks >= 0.9 * (double)(waves * cap)) {
            slices = t;
            break;
        }
    }
    if ((long long)slices * Sh > 0x7fffffffLL) return HC_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)(slices * Sh), Co);
    uint2* pc = reinterpret_cast<uint2*>(pieces);
    if (gelu_y)
        bias_rows_kernel<true, true><<<grid, 256, 0, st>>>(gy, tmp, N, Co, Ho, Wo, S, own_w, Sh, own_h, (int)slices,
                                                           pc, ps / 4, gelu_y);
    else if (pieces)
        bias_rows_kernel<true, false><<<grid, 256, 0, st>>>(gy, tmp, N, Co, Ho, Wo, S, own_w, Sh, own_h, (int)slices,
                                                            pc, ps / 4, nullptr);
    else
        bias_rows_kernel<false, false><<<grid, 256, 0, st>>>(gy, tmp, N, Co, Ho, Wo, S, own_w, Sh, own_h,
                                                             (int)slices, nullptr, 0, nullptr);
    hc_status s = launched("bias_rows_kernel", st);
    if (s) return s;
    return launch_sum_rows(tmp, gbp, (int)slices, (long long)Sh * S * Co, st);  // slices in order
}

hc_status launch_sum_rows(const float* in, float* out, int rows, long long count, cudaStream_t st) {
    const int threads = 256;
    long long blocks = (count + threads - 1) / threads;
    if (blocks > 152LL * 16) blocks = 152LL * 16;
    if (blocks < 1) blocks = 1;
    sum_rows_kernel<<<(unsigned)blocks, threads, 0, st>>>(in, out, rows, count);
    return launched("sum_rows_kernel", st);
}

}  // namespace hc
