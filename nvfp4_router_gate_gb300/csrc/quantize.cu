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
#include "nvr_tcgen05.cuh"

namespace nvr {

// The amax kernel's last CTA publishes the per-call quantizer record `qrec`:
// four words {gsa, RN(1/gsa), division mode (as int bits), amax}.

template <bool kBF16>
__global__ void __launch_bounds__(kAmaxThreads, 4)
amax_kernel(const void* __restrict__ x, int64_t n_vec16, uint32_t* __restrict__ partials,
            uint32_t* __restrict__ ticket, float* __restrict__ gsa_out, float* __restrict__ qrec) {
  const uint4* v = static_cast<const uint4*>(x);
  uint32_t m = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // eight independent 16-byte loads in flight per thread
  for (; i + 7 * stride < n_vec16; i += 8 * stride) {
    uint4 a[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) a[u] = __ldg(v + i + u * stride);
#pragma unroll
    for (int u = 0; u < 8; ++u) m = max(m, absmax_bits16B<kBF16>(a[u]));
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
    const QuantScale qs = make_quant_scale(amax);
    *gsa_out = qs.gsa;
    qrec[0] = qs.gsa;
    qrec[1] = qs.rgsa;
    qrec[2] = __int_as_float(qs.mode);
    qrec[3] = amax;
    *ticket = 0u;                          // ready for the next call
  }
}

// The same reduction fed by bulk copies: a persistent grid (one CTA per SM)
// streams 32 KB chunks through a 6-stage shared-memory ring (192 KB in flight
// per SM); one thread issues cp.async.bulk for the chunks ahead while all
// threads reduce the landed ones.  CTA b takes chunks b, b + G, b + 2G, ...
// (G CTAs): the refill of a stage needs no claim from a counter in memory,
// whose round trip to L2 per chunk halved the stream rate.  Bulk copies keep
// far more bytes in flight per SM than per-thread loads, which is what a pure
// HBM stream needs.  Waits on the ring are bounded (about a second); a
// timeout is recorded in the status word.
//
// Launched with programmatic dependent launch: the grid may become resident
// while the previous kernel of the stream finishes, but it waits for it
// (griddepcontrol.wait: completed, its writes visible) before it reads x --
// the previous kernel may be the one that produced x -- or touches the
// workspace.  Each CTA lets the next kernel launch once its share of x has
// been read.
constexpr int kAmaxChunk = 32 * 1024;
constexpr int kAmaxStages = 6;

template <bool kBF16>
__global__ void __launch_bounds__(kAmaxThreads, 1)
amax_bulk_kernel(const uint8_t* __restrict__ x, int64_t nbytes, uint32_t* __restrict__ partials,
                 uint32_t* __restrict__ ticket, float* __restrict__ gsa_out, float* __restrict__ qrec,
                 uint32_t* __restrict__ status) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[kAmaxStages];
  __shared__ uint32_t red[kAmaxThreads / 32];
  __shared__ bool last;
  const int64_t n_chunks = (nbytes + kAmaxChunk - 1) / kAmaxChunk;
  const int64_t my_n = n_chunks > blockIdx.x ? (n_chunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  auto issue = [&](int64_t j, int (&fills)[kAmaxStages]) {     // thread 0: this CTA's chunk j
    const int st = static_cast<int>(j % kAmaxStages);
    const int64_t off = (blockIdx.x + j * gridDim.x) * static_cast<int64_t>(kAmaxChunk);
    const uint32_t bytes = static_cast<uint32_t>(nbytes - off < kAmaxChunk ? nbytes - off : kAmaxChunk);
    ++fills[st];
    mbar_arrive_expect_tx(full + st, bytes);
    bulk_load(ring + st * kAmaxChunk, x + off, bytes, full + st);
  };
  int fills[kAmaxStages] = {0, 0, 0, 0, 0, 0};     // thread 0: copies issued per stage
  if (threadIdx.x == 0) {
    for (int st = 0; st < kAmaxStages; ++st) mbar_init(full + st, 1);
    fence_mbar_init();
  }
  // x and the workspace counters may be written by the previous kernel
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0)
    for (int64_t j = 0; j < kAmaxStages && j < my_n; ++j) issue(j, fills);
  __syncthreads();
  const uint64_t deadline = globaltimer_ns() + 1000000000ull;
  volatile int never = 0;
  uint32_t m = 0;
  bool ok = true;
  for (int64_t j = 0; j < my_n; ++j) {
    const int st = static_cast<int>(j % kAmaxStages);
    const uint32_t parity = static_cast<uint32_t>((j / kAmaxStages) & 1);
    ok = __syncthreads_and(mbar_wait(full + st, parity, deadline, &never)) != 0;
    if (!ok) break;
    const int64_t off = (blockIdx.x + j * gridDim.x) * static_cast<int64_t>(kAmaxChunk);
    const int nvec = static_cast<int>((nbytes - off < kAmaxChunk ? nbytes - off : kAmaxChunk) / 16);
    const uint4* v = reinterpret_cast<const uint4*>(ring + st * kAmaxChunk);
#pragma unroll 8
    for (int u = threadIdx.x; u < nvec; u += kAmaxThreads) m = max(m, absmax_bits16B<kBF16>(v[u]));
    __syncthreads();                               // the stage has been read
    if (threadIdx.x == 0 && j + kAmaxStages < my_n) issue(j + kAmaxStages, fills);
  }
  if (!ok) {
    // wait (bounded) for this CTA's copies still in flight, then give up
    if (threadIdx.x == 0) {
      report_timeout(status);
      const uint64_t drain = globaltimer_ns() + 1000000000ull;
      for (int st = 0; st < kAmaxStages; ++st) {
        if (fills[st] == 0) continue;
        // the latest fill of this stage completes phase fills - 1
        const uint32_t parity = static_cast<uint32_t>((fills[st] - 1) & 1);
        while (!mbar_try_wait(full + st, parity) && globaltimer_ns() < drain) {
        }
      }
    }
    __syncthreads();
    return;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0;
    for (int w = 0; w < kAmaxThreads / 32; ++w) b = max(b, red[w]);
    partials[blockIdx.x] = b;
    __threadfence();
    last = (atomicAdd(ticket, 1u) == gridDim.x - 1);
  }
  __syncthreads();
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
    const QuantScale qs = make_quant_scale(amax);
    *gsa_out = qs.gsa;
    qrec[0] = qs.gsa;
    qrec[1] = qs.rgsa;
    qrec[2] = __int_as_float(qs.mode);
    qrec[3] = amax;
    *ticket = 0u;                                  // ready for the next call
  }
}

// Two consecutive 16-element blocks of one row per thread: four (bf16) or
// eight (fp32) 16-byte loads, one 16-byte code store, two scale bytes.  Rows
// in [rows, rows_pad) only write zero scale bytes (tile layout padding).
template <bool kBF16, bool kTiled>
__global__ void __launch_bounds__(kQuantThreads)
quantize_kernel(const void* __restrict__ x, uint32_t rows, uint32_t rows_pad, uint32_t D,
                const float* __restrict__ qrec, uint8_t* __restrict__ codes,
                uint8_t* __restrict__ sf) {
  __shared__ float s_rcp[128];                 // RN(1 / dec(b)) for scale bytes b
  if (threadIdx.x < 128) {
    const uint32_t b = threadIdx.x;
    s_rcp[b] = (b >= 1 && b <= 126) ? __frcp_rn(e4m3_value(b)) : 0.0f;
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t KB = D / kBlock;
  const uint32_t pairs_per_row = KB / 2;
  const uint32_t g = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t r = g / pairs_per_row;
  const uint32_t c = 2 * (g - r * pairs_per_row);          // first block of the pair
  // no early return: every lane of the warp takes part in the shuffle below
  uint32_t b0 = 0, b1 = 0;
  if (r < rows) {
    QuantScale qs;
    qs.gsa = __ldg(qrec);
    qs.rgsa = __ldg(qrec + 1);
    qs.mode = __float_as_int(__ldg(qrec + 2));
    uint4 q;
    Block16 blk;
    const size_t e0 = static_cast<size_t>(r) * D + static_cast<size_t>(c) * kBlock;
    load_block16<kBF16>(x, e0, blk);
    b0 = quant_block16_bracket(blk, qs, q.x, q.y, s_rcp);
    load_block16<kBF16>(x, e0 + kBlock, blk);
    b1 = quant_block16_bracket(blk, qs, q.z, q.w, s_rcp);
    *reinterpret_cast<uint4*>(codes + static_cast<size_t>(r) * (D / 2) + static_cast<size_t>(c) * 8) = q;
  }
  if (kTiled) {
    // blocks 4c'..4c'+3 of a row are 4 consecutive bytes of one tile line:
    // the even lane of each pair of lanes writes them (KB % 4 == 0, so both
    // lanes hold the same row)
    const uint32_t o = __shfl_down_sync(0xFFFFFFFFu, b0 | (b1 << 8), 1);
    if ((c & 3) == 0 && r < rows_pad)
      *reinterpret_cast<uint32_t*>(sf + sf_tile_offset(r, c, KB)) = b0 | (b1 << 8) | (o << 16);
  } else if (r < rows) {
    *reinterpret_cast<uint16_t*>(sf + static_cast<size_t>(r) * KB + c) = static_cast<uint16_t>(b0 | (b1 << 8));
  }
}

// ------------------------------------------------------------------ launchers

cudaError_t launch_amax(const void* x, bool bf16, int64_t n_elems, uint32_t* partials,
                        uint32_t* ticket, float* gsa_out, float* qrec, int grid,
                        cudaStream_t s) {
  const int64_t n_vec16 = n_elems * (bf16 ? 2 : 4) / 16;
  if (bf16)
    amax_kernel<true><<<grid, kAmaxThreads, 0, s>>>(x, n_vec16, partials, ticket, gsa_out, qrec);
  else
    amax_kernel<false><<<grid, kAmaxThreads, 0, s>>>(x, n_vec16, partials, ticket, gsa_out, qrec);
  return cudaGetLastError();
}

cudaError_t launch_amax_bulk(const void* x, bool bf16, int64_t n_elems, uint32_t* partials,
                             uint32_t* ticket, float* gsa_out, float* qrec, uint32_t* status,
                             int grid, cudaStream_t s) {
  static bool attr_set[kMaxDevices][2] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const int smem = kAmaxStages * kAmaxChunk;
  if (!attr_set[dev][bf16]) {
    e = bf16 ? cudaFuncSetAttribute(amax_bulk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
             : cudaFuncSetAttribute(amax_bulk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev][bf16] = true;
  }
  const int64_t nbytes = n_elems * (bf16 ? 2 : 4);
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kAmaxThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16)
    return cudaLaunchKernelEx(&cfg, amax_bulk_kernel<true>, xb, nbytes, partials, ticket, gsa_out, qrec, status);
  return cudaLaunchKernelEx(&cfg, amax_bulk_kernel<false>, xb, nbytes, partials, ticket, gsa_out, qrec, status);
}

cudaError_t launch_quantize(const void* x, bool bf16, int64_t rows, int64_t D, bool tiled,
                            const float* qrec, uint8_t* codes, uint8_t* sf, cudaStream_t s) {
  const int64_t rows_pad = tiled ? (rows + 127) / 128 * 128 : rows;
  const int64_t n_threads = rows_pad * (D / kBlock / 2);
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
  const uint32_t r32 = static_cast<uint32_t>(rows), rp32 = static_cast<uint32_t>(rows_pad),
                 d32 = static_cast<uint32_t>(D);
  if (bf16 && tiled) return cudaLaunchKernelEx(&cfg, quantize_kernel<true, true>, x, r32, rp32, d32, qrec, codes, sf);
  if (bf16) return cudaLaunchKernelEx(&cfg, quantize_kernel<true, false>, x, r32, rp32, d32, qrec, codes, sf);
  if (tiled) return cudaLaunchKernelEx(&cfg, quantize_kernel<false, true>, x, r32, rp32, d32, qrec, codes, sf);
  return cudaLaunchKernelEx(&cfg, quantize_kernel<false, false>, x, r32, rp32, d32, qrec, codes, sf);
}

}  // namespace nvr
