// quantize.cu -- runtime NVFP4 quantization of a whole tensor (sm_103a).
//
// Source: "nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py",
// runtime-gsa section (gsa = max|x| / (6 * 448) from the actual activations),
// and "commit df05289: dsv4/layers/grouped_linear.py", zero-sync fused quantize
// section (one tensor, one global scale, computed and kept on the GPU; no
// .item() host sync).
//
// Two kernels, stream-ordered:
//   amax_kernel     -- |x| max: 16-byte loads, warp shuffles, a per-CTA partial
//                      in the workspace, and a last-CTA ticket that reduces the
//                      partials, writes gsa and resets the ticket.
//   quantize_kernel -- one thread per 16-element block: 32-byte (bf16) or
//                      64-byte (fp32) vector loads, the block quantizer shared
//                      with the decode kernel, packed 8-byte code stores, scale
//                      bytes in the linear or the 128x4 tile layout.
// The quantize kernel is launched with programmatic dependent launch and waits
// on the amax kernel's results with griddepcontrol.wait.
#include "nvr_internal.h"

namespace nvr {

template <bool kBF16>
__global__ void __launch_bounds__(kAmaxThreads)
amax_kernel(const void* __restrict__ x, int64_t n_vec16, uint32_t* __restrict__ partials,
            uint32_t* __restrict__ ticket, float* __restrict__ gsa_out, float* __restrict__ amax_out) {
  const uint4* v = static_cast<const uint4*>(x);
  uint32_t m = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // four independent loads in flight per thread
  for (; i + 3 * stride < n_vec16; i += 4 * stride) {
    const uint4 a = __ldg(v + i), b = __ldg(v + i + stride), c = __ldg(v + i + 2 * stride),
                d = __ldg(v + i + 3 * stride);
    m = max(m, max(max(absmax_bits16B<kBF16>(a), absmax_bits16B<kBF16>(b)),
                   max(absmax_bits16B<kBF16>(c), absmax_bits16B<kBF16>(d))));
  }
  for (; i < n_vec16; i += stride) m = max(m, absmax_bits16B<kBF16>(__ldg(v + i)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __shared__ uint32_t red[kAmaxThreads / 32];
  __shared__ bool last;
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0;
    for (int w = 0; w < kAmaxThreads / 32; ++w) b = max(b, red[w]);
    partials[blockIdx.x] = b;
    __threadfence();
    const uint32_t t = atomicAdd(ticket, 1u);
    last = (t == gridDim.x - 1);
  }
  __syncthreads();
  // let the dependent quantize kernel start its launch while the tail finishes
  asm volatile("griddepcontrol.launch_dependents;");
  if (!last) return;
  __threadfence();
  uint32_t b = 0;
  for (uint32_t j = threadIdx.x; j < gridDim.x; j += blockDim.x) b = max(b, __ldcg(partials + j));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) b = max(b, __shfl_xor_sync(0xFFFFFFFFu, b, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = b;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int w = 0; w < kAmaxThreads / 32; ++w) r = max(r, red[w]);
    const float amax = __uint_as_float(r);
    *gsa_out = __fdiv_rn(amax, kGsaDivisor);
    if (amax_out) *amax_out = amax;
    *ticket = 0u;                          // ready for the next call
  }
}

// One thread per (row, 16-element block).  Rows in [rows, rows_pad) only write
// zero scale bytes (tile layout padding).
template <bool kBF16, bool kTiled>
__global__ void __launch_bounds__(kQuantThreads)
quantize_kernel(const void* __restrict__ x, int64_t rows, int64_t rows_pad, int64_t D,
                const float* __restrict__ amax_in, uint8_t* __restrict__ codes,
                uint8_t* __restrict__ sf) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t KB = D / kBlock;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t r = g / KB, c = g - r * KB;
  // no early return: every lane of the warp takes part in the shuffles below
  uint32_t byte = 0;
  if (r < rows) {
    const QuantScale qs = make_quant_scale(__ldcg(amax_in));
    Block16 blk;
    load_block16<kBF16>(x, static_cast<size_t>(r * D + c * kBlock), blk);
    uint32_t lo, hi;
    byte = quant_block16(blk, qs, lo, hi);
    *reinterpret_cast<uint2*>(codes + r * (D / 2) + c * 8) = make_uint2(lo, hi);
  }
  if (kTiled) {
    // blocks 4c'..4c'+3 of a row are 4 consecutive bytes of one tile line:
    // gather them in the lane holding c % 4 == 0 (KB % 4 == 0, so the four
    // lanes always share the row)
    const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, byte, 1);
    const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, byte, 2);
    const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, byte, 3);
    if ((c & 3) == 0 && r < rows_pad)
      *reinterpret_cast<uint32_t*>(sf + sf_tile_offset(r, c, KB)) = byte | (b1 << 8) | (b2 << 16) | (b3 << 24);
  } else if (r < rows) {
    sf[r * KB + c] = static_cast<uint8_t>(byte);
  }
}

// ------------------------------------------------------------------ launchers

cudaError_t launch_amax(const void* x, bool bf16, int64_t n_elems, uint32_t* partials,
                        uint32_t* ticket, float* gsa_out, float* amax_out, int grid,
                        cudaStream_t s) {
  const int64_t n_vec16 = n_elems * (bf16 ? 2 : 4) / 16;
  if (bf16)
    amax_kernel<true><<<grid, kAmaxThreads, 0, s>>>(x, n_vec16, partials, ticket, gsa_out, amax_out);
  else
    amax_kernel<false><<<grid, kAmaxThreads, 0, s>>>(x, n_vec16, partials, ticket, gsa_out, amax_out);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const void* x, bool bf16, int64_t rows, int64_t D, bool tiled,
                            const float* amax, uint8_t* codes, uint8_t* sf, cudaStream_t s) {
  const int64_t rows_pad = tiled ? (rows + 127) / 128 * 128 : rows;
  const int64_t n_threads = rows_pad * (D / kBlock);
  const int64_t grid = (n_threads + kQuantThreads - 1) / kQuantThreads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kQuantThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16 && tiled) return cudaLaunchKernelEx(&cfg, quantize_kernel<true, true>, x, rows, rows_pad, D, amax, codes, sf);
  if (bf16) return cudaLaunchKernelEx(&cfg, quantize_kernel<true, false>, x, rows, rows_pad, D, amax, codes, sf);
  if (tiled) return cudaLaunchKernelEx(&cfg, quantize_kernel<false, true>, x, rows, rows_pad, D, amax, codes, sf);
  return cudaLaunchKernelEx(&cfg, quantize_kernel<false, false>, x, rows, rows_pad, D, amax, codes, sf);
}

}  // namespace nvr
