// Throughput of the plain ALU pipes the solver is bound by: FP32 FMA
// (scalar and packed f32x2) and FP64 FMA on the current GPU, for the
// context of the benchmark's roofline (the roofline's own peaks are derived
// from unit counts and the maximum clock).  Each thread runs 8 independent
// FMA chains; the grid is 8 blocks of 256 threads per SM; the best of six
// timed launches (CUDA events) after two untimed ones is reported.
// Also the latency of dependent chains, in SM cycles per link (one warp,
// clock64 around 4,096 links): a scalar FMA, a packed f32x2 FMA, a packed
// multiply, and one Givens rotation of a row pair (x, y) -> (c x + s y,
// c y - s x), packed and scalar, whose chain bounds the eigenvector update.
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

constexpr int kLinks = 4096;

__device__ __forceinline__ uint64_t pk2(float a, float b)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul2v(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm volatile("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2v(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// cyc[0..4]: cycles of kLinks links of each chain (lane 0 of one warp)
__global__ void chains(float *out, long long *cyc, float cs, float sn)
{
    const uint64_t c = pk2(cs, cs), s = pk2(sn, sn), ns = pk2(-sn, -sn);
    uint64_t x = pk2(threadIdx.x, 1.f), y = pk2(2.f, threadIdx.x * 0.5f);
    float fx = threadIdx.x, fy = 2.f;
    long long t0 = clock64();
    for (int i = 0; i < kLinks; ++i)
        fx = fmaf(cs, fx, sn);
    long long t1 = clock64();
    if (threadIdx.x == 0)
        cyc[0] = t1 - t0;
    t0 = clock64();
    for (int i = 0; i < kLinks; ++i)
        x = fma2v(c, x, s);
    t1 = clock64();
    if (threadIdx.x == 0)
        cyc[1] = t1 - t0;
    t0 = clock64();
    for (int i = 0; i < kLinks; ++i)
        x = mul2v(c, x);
    t1 = clock64();
    if (threadIdx.x == 0)
        cyc[2] = t1 - t0;
    t0 = clock64();
    for (int i = 0; i < kLinks; ++i) {
        const uint64_t xo = x;
        x = fma2v(c, x, mul2v(s, y));
        y = fma2v(c, y, mul2v(ns, xo));
        const uint64_t t = x;
        x = y;
        y = t;
    }
    t1 = clock64();
    if (threadIdx.x == 0)
        cyc[3] = t1 - t0;
    t0 = clock64();
    for (int i = 0; i < kLinks; ++i) {
        const float xo = fx;
        fx = fmaf(cs, fx, sn * fy);
        fy = fmaf(cs, fy, -sn * xo);
        const float t = fx;
        fx = fy;
        fy = t;
    }
    t1 = clock64();
    if (threadIdx.x == 0)
        cyc[4] = t1 - t0;
    float a, b, a2, b2;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a2), "=f"(b2) : "l"(y));
    out[threadIdx.x] = a + b + a2 + b2 + fx + fy;
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
    // dependent-chain latencies: one warp, the last of three launches
    long long *cyc = nullptr;
    if (cudaMalloc(&cyc, 5 * sizeof(long long)) != cudaSuccess)
        return 1;
    for (int r = 0; r < 3; ++r)
        chains<<<1, 32>>>(of, cyc, 0.6f, 0.8f);
    long long hc[5] = {0, 0, 0, 0, 0};
    if (cudaMemcpy(hc, cyc, sizeof(hc), cudaMemcpyDeviceToHost) != cudaSuccess)
        return 1;
    printf("{\"fp32_fma_tflops\": %.3f, \"fp32x2_fma_tflops\": %.3f, \"fp64_fma_tflops\": %.4f, "
           "\"sms\": %d, \"clock_attribute_khz\": %d, \"cycles_per_link\": {\"fma\": %.2f, "
           "\"fma_f32x2\": %.2f, \"mul_f32x2\": %.2f, \"rotation_f32x2\": %.2f, \"rotation_scalar\": %.2f}}\n",
           tflops[0], tflops[1], tflops[2], sms, clk, hc[0] / (double)kLinks, hc[1] / (double)kLinks,
           hc[2] / (double)kLinks, hc[3] / (double)kLinks, hc[4] / (double)kLinks);
    cudaFree(cyc);
    cudaFree(of);
    cudaFree(od);
    return 0;
}
