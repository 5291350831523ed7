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

// Bias-gradient partial sums, stage 1: block (slice, co, r) sums grad_output over
// its slice of the (n, i) rows and shard r's own output columns, in a fixed
// order (strided thread sums, then a shuffle tree and the warp sums in order).
// part[(slice * S + r) * Co + co].
__global__ void bias_slices_kernel(const float* __restrict__ gy, float* __restrict__ part, int N, int Co, int Ho,
                                   int Wo, int S, int own_w, int slices) {
    __shared__ float red[32];
    const int slice = blockIdx.x, co = blockIdx.y, r = blockIdx.z;
    const int j0 = r * own_w, j1 = (r == S - 1) ? Wo : j0 + own_w;
    const int nj = j1 - j0;
    const long long nrows = (long long)N * Ho;
    const long long r0 = nrows * slice / slices, r1 = nrows * (slice + 1) / slices;
    float acc = 0.0f;
    for (long long row = r0; row < r1; row++) {
        const int n = (int)(row / Ho), i = (int)(row % Ho);
        const float* p = gy + (((long long)n * Co + co) * Ho + i) * Wo + j0;
        for (int j = threadIdx.x; j < nj; j += blockDim.x) acc += __ldg(p + j);
    }
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int k = 0; k < (int)(blockDim.x >> 5); k++) t += red[k];
        part[((long long)slice * S + r) * Co + co] = t;
    }
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
    hc_status s = launched();
    if (s) return s;
    return launch_sum_rows(tmp, out, (rows + kColumnGroup - 1) / kColumnGroup, count, st);
}

size_t bias_grad_ws_floats(int Co, int S) { return (size_t)kBiasSlices * S * Co; }

hc_status launch_bias_grad_partials(const float* gy, float* gbp, int N, int Co, int Ho, int Wo, int S, int own_w,
                                    float* tmp, cudaStream_t st) {
    bias_slices_kernel<<<dim3(kBiasSlices, Co, S), 128, 0, st>>>(gy, tmp, N, Co, Ho, Wo, S, own_w, kBiasSlices);
    hc_status s = launched();
    if (s) return s;
    return launch_sum_rows(tmp, gbp, kBiasSlices, (long long)S * Co, st);  // slices in order
}

hc_status launch_sum_rows(const float* in, float* out, int rows, long long count, cudaStream_t st) {
    const int threads = 256;
    long long blocks = (count + threads - 1) / threads;
    if (blocks > 152LL * 16) blocks = 152LL * 16;
    if (blocks < 1) blocks = 1;
    sum_rows_kernel<<<(unsigned)blocks, threads, 0, st>>>(in, out, rows, count);
    return launched();
}

}  // namespace hc
