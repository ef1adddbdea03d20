// probes.cu -- measurement kernels for roofline denominators that the library's own kernels are
// judged against: the FP32 FMA rate of the CUDA cores and the read bandwidth of the L2 cache.
// They compute nothing for the method; the caller times them with CUDA events.
#include "common.cuh"
#include "kernels.cuh"

namespace csa {

// 16 independent FMA chains per thread, `iters` steps each: 32 * iters FLOP per thread. The
// chains' start values depend on the thread and the result is stored, so nothing folds away.
__global__ void __launch_bounds__(256) probe_ffma_kernel(int iters, float *out) {
    float x[16];
    const float a = 1.0f + 1e-7f * (float)(threadIdx.x & 7), c = 1e-7f;
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (float)(threadIdx.x + i) * 1e-3f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = fmaf(x[i], a, c);
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s += x[i];
    out[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// Reads n4 float4s `reps` times (grid-stride, 16-byte loads that may hit L2), one sum per CTA.
__global__ void __launch_bounds__(512) probe_read_kernel(const float4 *__restrict__ buf, int64_t n4, int reps,
                                                         float *out) {
    float acc = 0.0f;
    for (int r = 0; r < reps; ++r)
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
            const float4 v = __ldcg(buf + i);
            acc += (v.x + v.y) + (v.z + v.w);
        }
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) atomicAdd(out + blockIdx.x, acc);
}

void launch_probe_ffma(int blocks, int iters, float *out, cudaStream_t st) {
    probe_ffma_kernel<<<blocks, 256, 0, st>>>(iters, out);
    count_launches(1);
}

void launch_probe_read(const void *buf, int64_t bytes, int reps, int blocks, float *out, cudaStream_t st) {
    probe_read_kernel<<<blocks, 512, 0, st>>>(reinterpret_cast<const float4 *>(buf), bytes / 16, reps, out);
    count_launches(1);
}

}  // namespace csa
