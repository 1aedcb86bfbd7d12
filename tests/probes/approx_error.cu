// approx_error.cu -- test probe: the largest relative errors of the two
// hardware approximations the INT8 epilogue's fast path uses,
//   ex2.approx.ftz.f32 over every float y in [-116, 116] (2^y, |t| <= 80),
//   rcp.approx.ftz.f32 over every float d in [1, 2^116] (1 / (1 + e^-t)),
// each against the double-precision value.  Built and run by
// tests/test_hw_approx.py; not part of the library.
#include <cstdint>
#include <cuda_runtime.h>

__device__ unsigned long long g_worst[2];   // doubles >= 0 order like their bit patterns

__device__ __forceinline__ float key_to_float(long long k) {
    const uint32_t u = k < 0 ? (0x80000000u | (uint32_t)(-k)) : (uint32_t)k;
    return __uint_as_float(u);
}

__global__ void ex2_sweep(long long klo, long long khi) {
    double worst = 0.0;
    for (long long k = klo + blockIdx.x * (long long)blockDim.x + threadIdx.x; k <= khi;
         k += (long long)gridDim.x * blockDim.x) {
        const float y = key_to_float(k);
        float e;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(y));
        const double ref = exp2((double)y);
        const double err = fabs((double)e - ref) / ref;
        worst = err > worst ? err : worst;
    }
    atomicMax(&g_worst[0], (unsigned long long)__double_as_longlong(worst));
}

__global__ void rcp_sweep(uint32_t ulo, uint32_t uhi) {
    double worst = 0.0;
    for (uint32_t u = ulo + blockIdx.x * blockDim.x + threadIdx.x; u <= uhi && u >= ulo; u += gridDim.x * blockDim.x) {
        const float d = __uint_as_float(u);
        float r;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
        const double err = fabs((double)r * (double)d - 1.0);
        worst = err > worst ? err : worst;
    }
    atomicMax(&g_worst[1], (unsigned long long)__double_as_longlong(worst));
}

static long long float_key(float f) {
    uint32_t u;
    __builtin_memcpy(&u, &f, 4);
    return (u & 0x80000000u) ? -(long long)(u & 0x7fffffffu) : (long long)u;
}

extern "C" int approx_worst(double *ex2_err, double *rcp_err) {
    const unsigned long long zero[2] = {0ull, 0ull};
    if (cudaMemcpyToSymbol(g_worst, zero, sizeof(zero)) != cudaSuccess) return 1;
    ex2_sweep<<<1024, 256>>>(float_key(-116.0f), float_key(116.0f));
    uint32_t lo, hi;
    const float one = 1.0f, top = 0x1p116f;
    __builtin_memcpy(&lo, &one, 4);
    __builtin_memcpy(&hi, &top, 4);
    rcp_sweep<<<1024, 256>>>(lo, hi);
    if (cudaDeviceSynchronize() != cudaSuccess) return 2;
    unsigned long long w[2];
    if (cudaMemcpyFromSymbol(w, g_worst, sizeof(w)) != cudaSuccess) return 3;
    __builtin_memcpy(ex2_err, &w[0], 8);
    __builtin_memcpy(rcp_err, &w[1], 8);
    return 0;
}
