// gemm_splitk.cu -- the router for up to 256 experts: block-scaled NVFP4 gate
// GEMM on the 5th-generation tensor cores split along K over S CTAs, then a
// warp-per-token router epilogue (sm_103a).
//
// Source: "nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py"
// (NVFP4 gate GEMM on Blackwell tensor cores, fused router epilogue) and
// "commit e0f60b9: dsv4/kernels/router/__init__.py" (activation_topk: sigmoid,
// biased top-k, gather of the unbiased scores, renormalise, routed scaling).
//
// A router GEMM is short and deep (T x <=256 outputs, D = 7168), so one CTA
// per 128-token tile would leave most SMs idle.  The K stages are split over
// S CTAs per tile; each accumulates a 128 x N fp32 partial in tensor memory
// and stores it with TMA to the workspace (S x T x 256 fp32, which stays in
// L2 between the two kernels).  The epilogue kernel, launched with
// programmatic dependent launch, adds the S partials of a token in a fixed
// order (the result is deterministic), scales by gsa_x * gsa_w and selects.
//
// GEMM kernel, per CTA (320 threads):
//   warp 0     TMA producer: per stage of 256 K-elements the x tile (128 rows
//              x 128 bytes), the W tile (128 or 256 rows x 128 bytes), both
//              with 128-byte swizzle, and the scale slabs (4 atoms of 128 rows
//              x 4 scales for x, 4 per 128-expert half for W) into a 4-deep
//              shared-memory ring;
//   warps 2-5  scale stagers: each copies the stage's scale atoms into its own
//              32-lane quarter of tensor memory with tcgen05.st (the atom
//              line i of 16 bytes goes to lane i of every quarter, 4 columns),
//              then signals the MMA warp.  Register stores keep the scale
//              traffic off the tensor pipe, which otherwise serialises a
//              tcgen05.cp with the MMAs;
//   warp 1     MMA issuer: one tcgen05.mma.kind::mxf4nvf4 (M=128, N=128 or
//              256, K=64) per 64-element K step into one fp32 accumulator;
//   warps 2-9  after the last MMA: tcgen05.ld of the accumulator, 32 x 32
//              blocks staged in shared memory (128-byte swizzle) and TMA-stored
//              to the partial buffer.
// Tensor memory (512 columns): accumulator at columns 0-255; the scales of
// ring stage s at 256 + 48 s: x at +0 (4 columns per K step), W at +16
// (8 columns per K step: experts 0-127, then 128-255).
#include "nvr_splitk.cuh"

namespace nvr {

namespace {

constexpr int kKStages = 4;
constexpr int kKATile = 128 * 128;                  // 128 x rows x 128 bytes
constexpr int kKBTile = 256 * 128;                  // up to 256 W rows x 128 bytes
constexpr int kKSfa = 4 * 512;                      // 4 scale atoms
constexpr int kKSfb = 2 * 4 * 512;                  // 4 atoms per 128-expert half
constexpr int kKStageBytes = kKATile + kKBTile + kKSfa + kKSfb;
constexpr int kKRing = kKStages * kKStageBytes;
constexpr int kKSmem = kKRing + 1024 /*barriers*/ + 1024 /*align*/;
constexpr int kKThreads = 320;
constexpr int kEpiWarpsPerCta = 8;                  // epilogue kernel: one token per warp
static_assert(kKStageBytes % 1024 == 0, "stages keep 1024-byte alignment");
static_assert(8 * 8192 <= kKRing, "store staging fits the ring");

struct SplitKParams {
  CUtensorMap tmap_a;          // x codes [T, D/2] uint8, box 128 x 128
  CUtensorMap tmap_b;          // W codes [N, D/2] uint8, box 128 x (128 * n_half)
  CUtensorMap tmap_p;          // partials [S][T][256] fp32, box 32 x 32 x 1
  const uint8_t* sfa;          // x scales, tile layout
  const uint8_t* sfb;          // W scales, tile layout
  int T, D, n_half, S;
  uint32_t* status;
  int test_stall;              // test hook: the MMA issuer issues nothing
};

__global__ void __launch_bounds__(kKThreads, 1)
splitk_gemm_kernel(const __grid_constant__ SplitKParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kKRing);
  uint64_t* empty = full + kKStages;
  uint64_t* sf_full = empty + kKStages;
  uint64_t* acc_full = sf_full + kKStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  uint32_t filled_mask = 0, fill_bits = 0;          // producer: ring stages with a fill in flight
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x / p.S;
  const int rank = blockIdx.x - m_tile * p.S;
  const int KB = p.D / kBlock;
  const int n_st = (KB + 15) / 16;                   // stages of 256 K-elements
  const int st0 = (rank * n_st) / p.S;
  const int my_st = ((rank + 1) * n_st) / p.S - st0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
      mbar_init(sf_full + s, 4);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&p.tmap_a);
    tma_prefetch_map(&p.tmap_b);
    tma_prefetch_map(&p.tmap_p);
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // the quantize kernel before us (programmatic launch) must have finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint64_t deadline = globaltimer_ns() + 1000000000ull;   // 1 s

  bool acc_ok = true;     // epilogue warps: the accumulator is complete
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int s = 0; s < my_st; ++s) {
      const int ks = st0 + s;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty + stage, phase ^ 1u, deadline, abort_flag))) {
        ok = false;
        break;
      }
      const int nkk = min(4, KB / 4 - 4 * ks);
      uint8_t* a = smem + stage * kKStageBytes;
      uint8_t* b = a + kKATile;
      uint8_t* sa = b + kKBTile;
      uint8_t* sb = sa + kKSfa;
      if (elect_one()) {
        mbar_arrive_expect_tx(full + stage, static_cast<uint32_t>(kKATile + p.n_half * 128 * 128 +
                                                                  512 * nkk * (1 + p.n_half)));
        tma_load_2d(a, &p.tmap_a, ks * 128, m_tile * 128, full + stage);
        tma_load_2d(b, &p.tmap_b, ks * 128, 0, full + stage);
        bulk_load(sa, p.sfa + (static_cast<size_t>(m_tile) * (KB / 4) + 4 * ks) * 512, 512u * nkk,
                  full + stage);
        for (int h = 0; h < p.n_half; ++h)
          bulk_load(sb + h * 2048, p.sfb + (static_cast<size_t>(h) * (KB / 4) + 4 * ks) * 512, 512u * nkk,
                    full + stage);
      }
      __syncwarp();
      filled_mask |= 1u << stage;
      fill_bits = (fill_bits & ~(1u << stage)) | (phase << stage);
      if (++stage == kKStages) { stage = 0; phase ^= 1u; }
    }
    if (!ok && lane == 0) {
      report_timeout(p.status);
      *abort_flag = 1;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (!p.test_stall) {
      const uint32_t idesc = idesc_mxf4nvf4(128, 128 * p.n_half);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int s = 0; s < my_st; ++s) {
        // the scale stagers waited for the stage's copies before signalling
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(sf_full + stage, phase, deadline, abort_flag) &&
                                         mbar_wait(full + stage, phase, deadline, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int ks = st0 + s;
        const int nkk = min(4, KB / 4 - 4 * ks);
        const uint8_t* a = smem + stage * kKStageBytes;
        const uint8_t* b = a + kKATile;
        const uint32_t sf_t = tmem + 256 + stage * 48;
        if (elect_one()) {
          for (int kk = 0; kk < nkk; ++kk)
            tc_mma_nvf4(tmem, desc_kmajor_sw128(smem_u32(a + 32 * kk)), desc_kmajor_sw128(smem_u32(b + 32 * kk)),
                        idesc, sf_t + 4 * kk, sf_t + 16 + 8 * kk, (s | kk) != 0);
          tc_commit(empty + stage);
        }
        __syncwarp();
        if (++stage == kKStages) { stage = 0; phase ^= 1u; }
      }
      if (ok && my_st > 0 && elect_one()) tc_commit(acc_full);
      __syncwarp();
      if (!ok && lane == 0) {
        report_timeout(p.status);
        *abort_flag = 1;
      }
    }
  } else {
    if (warp < 6) {
      // ------------------------------------------------------ scale stagers
      // Warp w writes tensor-memory lanes 32*(w%4)..+31.  Lane i holds line i
      // (16 bytes) of every atom of the stage: scales of rows i, i+32, i+64,
      // i+96 (4 bytes each, one per 16-element block of the K step).
      const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int s = 0; s < my_st; ++s) {
        // A new fill of this stage implies that the MMAs which read the
        // stage's previous scales have completed (the producer waited for them).
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(full + stage, phase, deadline, abort_flag))) {
          ok = false;
          break;
        }
        const uint8_t* sa = smem + stage * kKStageBytes + kKATile + kKBTile;
        const uint8_t* sb = sa + kKSfa;
        uint32_t va[16], vb0[16], vb1[16];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint4 x = ld_shared_v4(sa + 512 * kk + 16 * lane);
          va[4 * kk] = x.x; va[4 * kk + 1] = x.y; va[4 * kk + 2] = x.z; va[4 * kk + 3] = x.w;
        }
        // W columns per K step: [experts 0-127 (4)][experts 128-255 (4)]
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t* dst = kk < 2 ? vb0 : vb1;
          const int o = 8 * (kk & 1);
          const uint4 x0 = ld_shared_v4(sb + 512 * kk + 16 * lane);
          const uint4 x1 = ld_shared_v4(sb + 2048 + 512 * kk + 16 * lane);
          dst[o] = x0.x; dst[o + 1] = x0.y; dst[o + 2] = x0.z; dst[o + 3] = x0.w;
          dst[o + 4] = x1.x; dst[o + 5] = x1.y; dst[o + 6] = x1.z; dst[o + 7] = x1.w;
        }
        const uint32_t t0 = tmem + lane_base + 256 + stage * 48;
        tmem_store16(t0, va);
        tmem_store16(t0 + 16, vb0);
        tmem_store16(t0 + 32, vb1);
        tmem_store_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sf_full + stage);
        if (++stage == kKStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok && lane == 0) {
        report_timeout(p.status);
        *abort_flag = 1;
      }
    }
    // --------------------------------------------- wait for the accumulator
    if (my_st > 0) {
      acc_ok = bar_and(1, 256, mbar_wait(acc_full, 0, deadline, abort_flag));
      if (!acc_ok && threadIdx.x == 64) {
        report_timeout(p.status);
        *abort_flag = 1;
      }
    }
    tc_fence_after();
    // ------------------------------------------ store the partial with TMA
    // (the ring is free: every fill has been consumed by an MMA)
    store_partial_tile(&p.tmap_p, smem, tmem, warp, lane, m_tile, rank, p.n_half, p.T, my_st > 0 && acc_ok);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The epilogue kernel may be scheduled once every CTA got here (it waits
  // for this grid to finish before reading the partials).  Triggering only
  // now spreads its CTAs evenly instead of piling them onto idle SMs.
  asm volatile("griddepcontrol.launch_dependents;");
  if (*abort_flag && threadIdx.x == 0) {
    // After an abort, copies issued by the producer may still be landing in
    // this CTA's shared memory: wait (bounded) for the latest fill of every
    // ring stage to complete before the CTA exits.
    const uint64_t drain = globaltimer_ns() + 1000000000ull;
    for (int s = 0; s < kKStages; ++s) {
      if (!((filled_mask >> s) & 1u)) continue;
      while (!mbar_try_wait(full + s, (fill_bits >> s) & 1u)) {
        if (globaltimer_ns() > drain) break;
      }
    }
  }
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------ router epilogue

struct EpiParams {
  const float* partials;       // [S][T][256] fp32
  const float* x_gsa;
  const float* w_gsa;
  const float* bias;           // [N] or null
  int T, N, S, k, raw;
  float routed_scaling;
  int32_t* out_ids;
  float* out_w;
  float* logits;               // logits mode: write [T, N] logits instead of the top-k
};

// One warp per token (see route_token in nvr_splitk.cuh).
__global__ void __launch_bounds__(kEpiWarpsPerCta * 32)
router_epilogue_kernel(const __grid_constant__ EpiParams p) {
  __shared__ float4 s_row[kEpiWarpsPerCta][kRouteSlot];   // each warp's token slot
  __shared__ __align__(16) uint8_t s_scr[kEpiWarpsPerCta][kRouteScratch];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kEpiWarpsPerCta + warp;
  TokenRouter rt;
  rt.init(p.bias, p.N, p.k, p.raw, p.routed_scaling, lane);
  // the GEMM kernel before us (programmatic launch) must have finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (t >= p.T) return;                              // whole warp
  const float gscale = __fmul_rn(__ldg(p.x_gsa), __ldg(p.w_gsa));
  const int64_t tt[1] = {t};
  rt.route<1, true>(p.partials, static_cast<size_t>(p.T) * 256, p.S, tt, gscale, s_row[warp], lane, p.out_ids,
                    p.out_w, p.logits, nullptr, s_scr[warp]);
}

}  // namespace

size_t splitk_partial_rows(int64_t T) {
  const int64_t rows_pad = (T + 127) / 128 * 128;
  const int64_t a = kMaxSplitK * rows_pad;
  const int64_t b = rows_pad > 256 * 128 ? rows_pad : 256 * 128;
  return static_cast<size_t>(a < b ? a : b);
}

int plan_splitk(int64_t T, int64_t D, int num_sms) {
  const int64_t m_tiles = (T + 127) / 128;
  const int64_t n_st = (D / kBlock + 15) / 16;
  int64_t S = num_sms / (m_tiles > 0 ? m_tiles : 1);
  if (S > kMaxSplitK) S = kMaxSplitK;
  if (S > n_st) S = n_st;
  if (S < 1) S = 1;
  const int64_t cap = static_cast<int64_t>(splitk_partial_rows(T)) / (m_tiles * 128);
  if (S > cap) S = cap;
  return static_cast<int>(S);
}

nvr_status launch_splitk_gemm(const uint8_t* x_codes, const uint8_t* x_sf, int64_t T, int64_t D,
                              const uint8_t* W_codes, const uint8_t* W_sf, int64_t N, float* partials,
                              uint32_t* status, int S, bool test_stall, cudaStream_t s) {
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVR_ERR_CUDA;
  if (N > 256 || S < 1 || S > kMaxSplitK) return NVR_ERR_UNSUPPORTED;
  if (static_cast<size_t>(S) * static_cast<size_t>((T + 127) / 128 * 128) > splitk_partial_rows(T))
    return NVR_ERR_UNSUPPORTED;
  if (!attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(splitk_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kKSmem);
    if (e != cudaSuccess) return cuda_status(e);
    attr_set[dev] = true;
  }
  SplitKParams g;
  const int n_half = N > 128 ? 2 : 1;
  if (!encode_codes(&g.tmap_a, x_codes, T, D, 128)) return NVR_ERR_UNSUPPORTED;
  if (!encode_codes(&g.tmap_b, W_codes, N, D, 128u * n_half)) return NVR_ERR_UNSUPPORTED;
  if (!encode_partials(&g.tmap_p, partials, T, S)) return NVR_ERR_UNSUPPORTED;
  g.sfa = x_sf; g.sfb = W_sf;
  g.T = static_cast<int>(T); g.D = static_cast<int>(D); g.n_half = n_half; g.S = S;
  g.status = status; g.test_stall = test_stall ? 1 : 0;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((T + 127) / 128 * S));
  cfg.blockDim = dim3(kKThreads);
  cfg.dynamicSmemBytes = kKSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, splitk_gemm_kernel, g));
}

nvr_status launch_router_epilogue(const float* partials, int S, const float* x_gsa, const float* w_gsa,
                                  int64_t T, int64_t N, const float* bias, int k, float routed_scaling,
                                  bool raw, int32_t* out_ids, float* out_w, float* logits, cudaStream_t s) {
  if (N > 256 || k > kMaxKmax || S < 1) return NVR_ERR_UNSUPPORTED;
  EpiParams e;
  e.partials = partials; e.x_gsa = x_gsa; e.w_gsa = w_gsa; e.bias = raw ? nullptr : bias;
  e.T = static_cast<int>(T); e.N = static_cast<int>(N); e.S = S; e.k = k; e.raw = raw ? 1 : 0;
  e.routed_scaling = routed_scaling; e.out_ids = out_ids; e.out_w = out_w; e.logits = logits;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((T + kEpiWarpsPerCta - 1) / kEpiWarpsPerCta));
  cfg.blockDim = dim3(kEpiWarpsPerCta * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, router_epilogue_kernel, e));
}

}  // namespace nvr
