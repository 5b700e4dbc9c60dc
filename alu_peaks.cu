// Throughput of the plain ALU pipes the solver is bound by: FP32 FMA
// (scalar and packed f32x2) and FP64 FMA on the current GPU, for the
// context of the benchmark's roofline (the roofline's own peaks are derived
// from unit counts and the maximum clock).  Each thread runs 8 independent
// FMA chains; the grid is 8 blocks of 256 threads per SM; the best of six
// timed launches (CUDA events) after two untimed ones is reported.
// Built and run by `python bench.py --alu-peaks`; prints one JSON line.
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

namespace {

constexpr int kIters = 4096;
constexpr int kChains = 8;

__global__ void fma_f32(float *out, float b, float c)
{
    float a[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i)
        a[i] = threadIdx.x * 1e-3f + i;
    for (int it = 0; it < kIters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i)
            a[i] = fmaf(a[i], b, c);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i)
        s += a[i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void fma_f32x2(float *out, float b, float c)
{
    uint64_t a[kChains], bb, cc;
    asm("mov.b64 %0, {%1, %2};" : "=l"(bb) : "f"(b), "f"(b));
    asm("mov.b64 %0, {%1, %2};" : "=l"(cc) : "f"(c), "f"(c));
#pragma unroll
    for (int i = 0; i < kChains; ++i) {
        const float x = threadIdx.x * 1e-3f + i;
        asm("mov.b64 %0, {%1, %2};" : "=l"(a[i]) : "f"(x), "f"(x + 0.5f));
    }
    for (int it = 0; it < kIters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i)
            asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(a[i]) : "l"(bb), "l"(cc));
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) {
        float x, y;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(a[i]));
        s += x + y;
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void fma_f64(double *out, double b, double c)
{
    double a[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i)
        a[i] = threadIdx.x * 1e-3 + i;
    for (int it = 0; it < kIters / 8; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i)
            a[i] = fma(a[i], b, c);
    }
    double s = 0.0;
#pragma unroll
    for (int i = 0; i < kChains; ++i)
        s += a[i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

int main()
{
    int dev = 0, sms = 0, clk = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&clk, cudaDevAttrClockRate, dev);
    const int blocks = sms * 8, threads = 256;
    const double nthreads = (double)blocks * threads;
    float *of = nullptr;
    double *od = nullptr;
    if (cudaMalloc(&of, (size_t)nthreads * sizeof(float)) != cudaSuccess ||
        cudaMalloc(&od, (size_t)nthreads * sizeof(double)) != cudaSuccess)
        return 1;
    cudaEvent_t s, t;
    cudaEventCreate(&s);
    cudaEventCreate(&t);
    double tflops[3];
    for (int k = 0; k < 3; ++k) {
        float best = 1e30f;
        for (int rep = 0; rep < 8; ++rep) {
            cudaEventRecord(s);
            if (k == 0)
                fma_f32<<<blocks, threads>>>(of, 0.999f, 1e-4f);
            else if (k == 1)
                fma_f32x2<<<blocks, threads>>>(of, 0.999f, 1e-4f);
            else
                fma_f64<<<blocks, threads>>>(od, 0.999, 1e-4);
            cudaEventRecord(t);
            cudaEventSynchronize(t);
            float ms = 0;
            cudaEventElapsedTime(&ms, s, t);
            if (rep > 1 && ms < best)
                best = ms;
        }
        if (cudaGetLastError() != cudaSuccess)
            return 1;
        const double fmas = nthreads * kChains * (k == 2 ? kIters / 8 : kIters) * (k == 1 ? 2 : 1);
        tflops[k] = 2.0 * fmas / (best * 1e-3) / 1e12;
    }
    printf("{\"fp32_fma_tflops\": %.3f, \"fp32x2_fma_tflops\": %.3f, \"fp64_fma_tflops\": %.4f, "
           "\"sms\": %d, \"clock_attribute_khz\": %d}\n",
           tflops[0], tflops[1], tflops[2], sms, clk);
    cudaFree(of);
    cudaFree(od);
    return 0;
}
