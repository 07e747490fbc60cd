// spec_selftest_ex2: re-measures the relative error of the hardware
// exponential (ex2.approx.ftz.f32) that the full-vocabulary path's certified
// fp32 draw relies on, exhaustively over every fp32 input in [-126, 1],
// against fp64.  The draw's error model uses 1.5e-7; this is its check.
#include <cstdint>

#include "spec_verify.h"

namespace {

__device__ unsigned g_ex2_worst;  // bit pattern of the largest relative error seen

__device__ __forceinline__ float ex2_hw(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// inputs: bit patterns [lo, hi) with the given sign bit
__global__ void ex2_scan(uint32_t lo, uint32_t hi, uint32_t sign) {
    const uint64_t n = (uint64_t)hi - lo;
    float worst = 0.0f;
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
        const float x = __uint_as_float((lo + (uint32_t)i) | sign);
        const double e = exp2((double)x);
        const float rel = (float)(fabs((double)ex2_hw(x) - e) / e);
        worst = fmaxf(worst, rel);
    }
    atomicMax(&g_ex2_worst, __float_as_uint(worst));  // non-negative floats order as integers
}

}  // namespace

extern "C" int spec_selftest_ex2(float *max_rel_err) {
    if (!max_rel_err) return SPEC_ERR_INVALID_ARG;
    const unsigned zero = 0u;
    cudaError_t e = cudaMemcpyToSymbol(g_ex2_worst, &zero, sizeof zero);
    if (e == cudaSuccess) {
        ex2_scan<<<1024, 256>>>(0u, 0x42FC0000u + 1u, 0x80000000u);  // [-126, -0]
        ex2_scan<<<1024, 256>>>(0u, 0x3F800000u + 1u, 0u);           // [0, 1]
        e = cudaGetLastError();
    }
    unsigned bits = 0u;
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&bits, g_ex2_worst, sizeof bits);  // synchronises
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
    *max_rel_err = __builtin_bit_cast(float, bits);
    return SPEC_OK;
}
