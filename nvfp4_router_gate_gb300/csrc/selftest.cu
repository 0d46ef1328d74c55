// selftest.cu -- an exhaustive check of the two hardware conversions every
// quantizer path relies on: cvt.rn.satfinite.e2m1x2.f32 (the E2M1 codes) and
// cvt.rn.satfinite.e4m3x2.f32 (the E4M3 block scales), over every float32
// bit pattern but the NaNs.
//
// Source: the formats' definitions and their maxima (6 for E2M1, 448 for the
// E4M3 scale; "nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py",
// runtime-gsa section): round to nearest with ties to the even code,
// saturation at the largest finite value.  Both conversions are monotone step
// functions of the magnitude, so the caller describes each by its rounding
// thresholds -- t_i, the smallest float32 bit pattern whose magnitude code is
// at least i -- and the kernel compares every conversion with the code the
// thresholds give: #{i : bits(|x|) >= t_i}, the sign bit set for a negative x
// with a nonzero code.  The sign of a zero result is not compared (the E2M1
// conversion returns +0 for a negative value that rounds to zero; the
// quantizers restore the sign from the input where it is visible).
#include "nvr_internal.h"

namespace nvr {

namespace {

constexpr int kSweepThreads = 256;

__device__ __forceinline__ uint32_t cvt_e2m1x2(float hi, float lo) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\t"
      "mov.b32 %0, {b, 0, 0, 0};\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
  return h;
}

// counts[0]: E2M1 mismatches, counts[1]: E4M3 mismatches, counts[2]: inputs
// checked; first[0..1]: the smallest mismatching bit pattern of each.
__global__ void __launch_bounds__(kSweepThreads)
conversion_sweep_kernel(const uint32_t* __restrict__ th2, const uint32_t* __restrict__ th8,
                        unsigned long long* __restrict__ counts, uint32_t* __restrict__ first) {
  __shared__ uint32_t s2[7], s8[128];
  if (threadIdx.x < 7) s2[threadIdx.x] = th2[threadIdx.x];
  if (threadIdx.x < 126) s8[threadIdx.x] = th8[threadIdx.x];
  if (threadIdx.x == 126 || threadIdx.x == 127) s8[threadIdx.x] = 0xFFFFFFFFu;   // above every magnitude
  __syncthreads();
  unsigned long long bad2 = 0, bad8 = 0, checked = 0;
  uint32_t f2 = 0xFFFFFFFFu, f8 = 0xFFFFFFFFu;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t u = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < (1ull << 32); u += stride) {
    const uint32_t b = static_cast<uint32_t>(u);
    const uint32_t mag = b & 0x7FFFFFFFu, neg = b >> 31;
    if (mag > 0x7F800000u) continue;                 // NaN: outside the quantizers' contract
    ++checked;
    const float x = __uint_as_float(b);
    uint32_t e2 = 0;
#pragma unroll
    for (int i = 0; i < 7; ++i) e2 += mag >= s2[i] ? 1u : 0u;
    uint32_t e8 = 0;                                 // #{i : s8[i] <= mag}, s8 ascending
#pragma unroll
    for (uint32_t step = 64; step >= 1; step >>= 1)
      if (s8[e8 + step - 1] <= mag) e8 += step;
    // the value in both halves of each paired conversion
    const uint32_t c2 = cvt_e2m1x2(x, x), c8 = cvt_e4m3x2(x, x);
    bool ok2 = true, ok8 = true;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t n = (c2 >> (4 * h)) & 0xFu, y = (c8 >> (8 * h)) & 0xFFu;
      ok2 = ok2 && (n & 7u) == e2 && (e2 == 0 || (n >> 3) == neg);
      ok8 = ok8 && (y & 0x7Fu) == e8 && (e8 == 0 || (y >> 7) == neg);
    }
    if (!ok2) { ++bad2; f2 = min(f2, b); }
    if (!ok8) { ++bad8; f8 = min(f8, b); }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    bad2 += __shfl_xor_sync(0xFFFFFFFFu, bad2, o);
    bad8 += __shfl_xor_sync(0xFFFFFFFFu, bad8, o);
    checked += __shfl_xor_sync(0xFFFFFFFFu, checked, o);
    f2 = min(f2, __shfl_xor_sync(0xFFFFFFFFu, f2, o));
    f8 = min(f8, __shfl_xor_sync(0xFFFFFFFFu, f8, o));
  }
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(counts, bad2);
    atomicAdd(counts + 1, bad8);
    atomicAdd(counts + 2, checked);
    atomicMin(first, f2);
    atomicMin(first + 1, f8);
  }
}

}  // namespace

}  // namespace nvr

using namespace nvr;

extern "C" nvr_status nvr_test_conversion_sweep(const uint32_t* th_e2m1, const uint32_t* th_e4m3,
                                                unsigned long long* counts, uint32_t* first, nvr_stream_t stream) {
  if (!th_e2m1 || !th_e4m3 || !counts || !first) return NVR_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(counts, 0, 3 * sizeof(unsigned long long), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(first, 0xFF, 2 * sizeof(uint32_t), s);
  if (e != cudaSuccess) return cuda_status(e);
  const int sms = device_sm_count();
  if (sms <= 0) return NVR_ERR_CUDA;
  conversion_sweep_kernel<<<sms * 8, kSweepThreads, 0, s>>>(th_e2m1, th_e4m3, counts, first);
  return cuda_status(cudaGetLastError());
}
