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

}  // namespace

hc_status launch_sum_rows(const float* in, float* out, int rows, long long count, cudaStream_t st) {
    const int threads = 256;
    long long blocks = (count + threads - 1) / threads;
    if (blocks > 152LL * 16) blocks = 152LL * 16;
    if (blocks < 1) blocks = 1;
    sum_rows_kernel<<<(unsigned)blocks, threads, 0, st>>>(in, out, rows, count);
    return launched();
}

}  // namespace hc
