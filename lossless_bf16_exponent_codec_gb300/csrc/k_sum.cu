// k_sum.cu -- the local step of a compressed reduce-scatter (ZipCCL digest
// 3.2, zipcclReduceScatter: an all-to-all of compressed chunks, then local
// decompression and a sum in higher precision).
//
// acc[i] = (first ? 0 : acc[i]) + (float)x[i] with x raw BF16 bits: the
// conversion is exact (bits << 16) and each element takes one IEEE
// single-precision addition, so W calls in source order give the bits of a
// sequential float32 sum in that order.  HBM-bound: 2 bytes in and 4 (or 8)
// bytes of accumulator per value; 8 values per thread and step, grid-stride.
#include "ez_internal.h"
#include "ez_common.cuh"

namespace ezk {
using namespace ez;

__global__ void __launch_bounds__(kThreads) k_accumulate_bf16(float* __restrict__ acc,
                                                             const uint16_t* __restrict__ x,
                                                             uint64_t n, int first)
{
    const uint64_t n8 = n / 8;
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    for (uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < n8; i += stride) {
        const uint4 w = ld_v4_nc(x + 8 * i);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        float4* a = reinterpret_cast<float4*>(acc + 8 * i);
        float4 lo = first ? make_float4(0.f, 0.f, 0.f, 0.f) : a[0];
        float4 hi = first ? make_float4(0.f, 0.f, 0.f, 0.f) : a[1];
        lo.x = __fadd_rn(lo.x, __uint_as_float(ws[0] << 16));
        lo.y = __fadd_rn(lo.y, __uint_as_float(ws[0] & 0xFFFF0000u));
        lo.z = __fadd_rn(lo.z, __uint_as_float(ws[1] << 16));
        lo.w = __fadd_rn(lo.w, __uint_as_float(ws[1] & 0xFFFF0000u));
        hi.x = __fadd_rn(hi.x, __uint_as_float(ws[2] << 16));
        hi.y = __fadd_rn(hi.y, __uint_as_float(ws[2] & 0xFFFF0000u));
        hi.z = __fadd_rn(hi.z, __uint_as_float(ws[3] << 16));
        hi.w = __fadd_rn(hi.w, __uint_as_float(ws[3] & 0xFFFF0000u));
        a[0] = lo;
        a[1] = hi;
    }
    // the tail (fewer than 8 values) in the first CTA
    if (blockIdx.x == 0 && threadIdx.x < n - 8 * n8) {
        const uint64_t j = 8 * n8 + threadIdx.x;
        const float v = __uint_as_float((uint32_t)x[j] << 16);
        acc[j] = first ? __fadd_rn(0.f, v) : __fadd_rn(acc[j], v);
    }
}

cudaError_t launch_accumulate_bf16(float* acc, const uint16_t* x, uint64_t n, int first, cudaStream_t s)
{
    if (!n) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const uint64_t want = cdiv(n / 8 ? n / 8 : 1, kThreads);
    const unsigned grid = (unsigned)umin64(want, (uint64_t)sms * 8);
    k_accumulate_bf16<<<grid, kThreads, 0, s>>>(acc, x, n, first);
    return cudaGetLastError();
}

}  // namespace ezk
