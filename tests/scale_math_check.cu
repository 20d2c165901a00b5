// Exhaustive check of the group-scale arithmetic in quant.cuh against the IEEE
// operations it replaces: group_scale<BITS> (fp16_rn of the correctly rounded
// amax / Q) for every non-negative finite fp32 amax, Q = 7 and 127, and
// scale_reciprocal (fl(1/s)) for every positive finite fp16 s.  Prints the
// mismatch counts; exits non-zero on any mismatch or CUDA error.
#include <cstdio>

#include "quant.cuh"

__device__ unsigned long long g_bad[3];

template <int BITS>
__global__ void scale_check(int slot) {
    const unsigned long long total = 0x7F800000ull;  // bit patterns of the finite non-negative fp32 values
    for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < total;
         i += (unsigned long long)gridDim.x * blockDim.x) {
        const float amax = __uint_as_float(static_cast<unsigned int>(i));
        uint16_t bits;
        kvq::group_scale<BITS>(amax, bits);
        const uint16_t ref = __half_as_ushort(__float2half_rn(__fdiv_rn(amax, static_cast<float>(kvq::QMax<BITS>::v))));
        if (bits != ref) atomicAdd(&g_bad[slot], 1ull);
    }
}

__global__ void reciprocal_check() {
    const unsigned int i = blockIdx.x * blockDim.x + threadIdx.x;  // fp16 bit pattern
    if (i == 0 || i >= 0x7C00u) return;
    const float s = __half2float(__ushort_as_half(static_cast<unsigned short>(i)));
    if (__float_as_uint(kvq::scale_reciprocal(s)) != __float_as_uint(__frcp_rn(s))) atomicAdd(&g_bad[2], 1ull);
}

int main() {
    const unsigned long long zero[3] = {0, 0, 0};
    cudaMemcpyToSymbol(g_bad, zero, sizeof(zero));
    scale_check<4><<<152 * 16, 256>>>(0);
    scale_check<8><<<152 * 16, 256>>>(1);
    reciprocal_check<<<(0x7C00 + 255) / 256, 256>>>();
    const cudaError_t e = cudaDeviceSynchronize();
    unsigned long long bad[3];
    cudaMemcpyFromSymbol(bad, g_bad, sizeof(bad));
    printf("cuda %s; group_scale Q=7 mismatches %llu; Q=127 mismatches %llu; scale_reciprocal mismatches %llu\n",
           cudaGetErrorString(e), bad[0], bad[1], bad[2]);
    return (e == cudaSuccess && bad[0] == 0 && bad[1] == 0 && bad[2] == 0) ? 0 : 1;
}
