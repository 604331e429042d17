// quant8.cu -- row-wise e4m3 quantization for the 8-bit GEMM variant.
//
// The variant follows the activation-quantized path of "Eager GPU Offload
// Without A Compute Graph", section "F16 and GGUF quantized linears"
// (quantize each activation tile once, run the MMA on 8-bit operands):
// on this GPU the 8-bit operands are e4m3 floats with one binary32 scale
// per row.  A row of f16 values v gets
//
//     amax = max |v|,  s = RN32(amax / 448),  inv = RN32(448 / amax)
//     code = e4m3(RN32(v * inv))     (round to nearest even, clamp to 448)
//
// with s = inv = 1 for an all-zero row; the code stands for code * s.
// Weights are quantized once (per output row, from their f16 cache) and
// activations once per call (per token).  Inputs are assumed finite.
//
// One warp per row, two passes over it: the largest magnitude (an integer
// max over the f16 magnitude bits, whose order is the order of the values),
// then the codes, eight per lane per step (a 16-byte load, an 8-byte store).
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "mq_internal.h"
#include "mq_launch.cuh"
#include "mq_ptx.cuh"

namespace mq {
namespace {

constexpr int kQThreads = 256;
constexpr int kRowsPerCta = kQThreads / 32;

__global__ void __launch_bounds__(kQThreads) k_quant_e4m3(const __half *__restrict__ src, int64_t rows, int64_t K,
                                                         int64_t ld, uint8_t *__restrict__ dst, int64_t ldo,
                                                         float *__restrict__ scales)
{
    grid_dep_launch();
    grid_dep_wait();   // the rows may come from the previous kernel on the stream
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + warp;
    if (r >= rows)
        return;
    const __half *row = src + r * ld;
    uint32_t mag = 0;   // two f16 magnitudes, max so far
    for (int64_t k = 8 * lane; k < K; k += 256) {
        const uint4 v = ldg_nc_v4(row + k);
        mag = __vmaxu2(mag, v.x & 0x7FFF7FFFu);
        mag = __vmaxu2(mag, v.y & 0x7FFF7FFFu);
        mag = __vmaxu2(mag, v.z & 0x7FFF7FFFu);
        mag = __vmaxu2(mag, v.w & 0x7FFF7FFFu);
    }
    const uint32_t m1 = (mag & 0xFFFFu) > (mag >> 16) ? (mag & 0xFFFFu) : (mag >> 16);
    const uint32_t mbits = __reduce_max_sync(0xFFFFFFFFu, m1);
    const float amax = __half2float(__ushort_as_half(static_cast<unsigned short>(mbits)));
    float s = 1.0f, inv = 1.0f;
    if (amax > 0.0f) {
        s = __fdiv_rn(amax, 448.0f);
        inv = __fdiv_rn(448.0f, amax);
    }
    uint8_t *out = dst + r * ldo;
    for (int64_t k = 8 * lane; k < K; k += 256) {
        const uint4 v = ldg_nc_v4(row + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t c[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            c[i] = cvt_e4m3x2(__fmul_rn(f.x, inv), __fmul_rn(f.y, inv));
        }
        *reinterpret_cast<uint2 *>(out + k) = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    }
    if (lane == 0)
        scales[r] = s;
}

}  // namespace

cudaError_t launch_quant_e4m3(const __half *src, int64_t rows, int64_t K, int64_t ld, uint8_t *dst, int64_t ldo,
                              float *scales, cudaStream_t s)
{
    if (rows <= 0)
        return cudaSuccess;
    if (K % 16 != 0 || ld % 8 != 0 || ldo % 16 != 0)
        return cudaErrorInvalidValue;
    const int64_t grid = (rows + kRowsPerCta - 1) / kRowsPerCta;
    if (grid > 0x7FFFFFFF)
        return cudaErrorInvalidValue;
    const cudaError_t e = launch_kernel(k_quant_e4m3, dim3(static_cast<unsigned>(grid)), dim3(kQThreads), 0, s, src,
                                        rows, K, ld, dst, ldo, scales);
    note_launch();
    return e;
}

}  // namespace mq
