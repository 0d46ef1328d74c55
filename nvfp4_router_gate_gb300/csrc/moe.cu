// moe.cu -- the NVFP4 grouped expert GEMM that consumes the router's output
// (expert ids per token), and the weighted combine of the expert outputs
// (sm_103a).
//
// Source: "nvfp4-megamoe-kernel commit df05289: dsv4/layers/grouped_linear.py"
// (grouped NVFP4 linear: one weight per group, the groups' rows flattened into
// one activation tensor quantized with one runtime global scale in one pass,
// expert offsets computed on the GPU with no host round trip, pre-allocated
// buffers) and the runtime-gsa section of "commit 04cf8ca:
// dsv4/layers/router.py" (the same runtime gsa in Nvfp4GroupedLinear and
// Nvfp4MoE).
//
// One call, four kernels chained with programmatic dependent launch, no host
// synchronisation and no allocation:
//   amax             x's runtime gsa (x once: the k copies of a token routed
//                    to k experts share x's max|x|);
//   moe_route        one CTA: expert counts (warp-aggregated shared-memory
//                    atomics), each expert's segment of rows padded to a
//                    multiple of 128, the list of (expert, 128-row token tile)
//                    work units and every routed pair's row -- the expert
//                    offsets stay on the GPU;
//   moe_quantize_scatter  x's NVFP4 codes and scale bytes (the standalone
//                    quantizer's arithmetic), each block quantized once and
//                    stored into the token's k segment rows, scales in the
//                    tensor-core tile layout;
//   moe_gemm         the weight-streaming GEMM of gemm_stream.cu per work unit:
//                    the expert's 128-row weight tiles are the MMA's M, the
//                    unit's 128 token rows its N; the epilogue stores
//                    y[t, j, n] for the unit's rows (fp32 or bf16).
// moe_combine (its own entry point) forms out[t] = sum_j w[t, j] y[t, j].
#include "nvr_splitk.cuh"

namespace nvr {

namespace {

constexpr int kRouteThreads = 1024;
constexpr int kMoeMaxExperts = 1024;
constexpr int kMThreads = 320;                  // producer, MMA, 8 epilogue warps
constexpr int kMEpi = 256;
constexpr int kMStages = 6;
constexpr int kMTile = 128 * 128;               // 128 rows x 128 bytes of codes
constexpr int kMSlab = 4 * 512;                 // 4 scale atoms
constexpr int kMStage = 2 * kMTile + 2 * kMSlab;
constexpr int kMSmem = kMStages * kMStage + 512 /*rows*/ + 1024 /*barriers*/ + 1024 /*align*/;
static_assert(kMStage % 1024 == 0 && kMSmem <= 227 * 1024, "shared-memory plan");

// --------------------------------------------------------------- routing
// Each routed pair's rank inside its expert's group (ids outside [0, E): -1),
// the segments (start, count), the work units; ctl[0]: work units, ctl[1]:
// rows of all segments.
__global__ void __launch_bounds__(kRouteThreads)
moe_route_kernel(const int32_t* __restrict__ ids, int n_pairs, int E, int32_t* __restrict__ rank_of_pair,
                 uint32_t* __restrict__ seg_start, uint32_t* __restrict__ seg_count, uint32_t* __restrict__ units,
                 uint32_t* __restrict__ ctl) {
  __shared__ uint32_t cnt[kMoeMaxExperts];
  __shared__ uint32_t wpad[32], wtile[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the ids may come from the router kernel just before
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  for (int e = tid; e < E; e += kRouteThreads) cnt[e] = 0u;
  __syncthreads();
  // each routed pair's rank inside its expert's group (the order inside a
  // group does not affect any output row); the ids are read as 16-byte
  // vectors, eight per thread in flight at once (ids and pos_of are 16-byte
  // aligned: checked on the host)
  const int n4 = n_pairs / 4;
  const int4* ids4 = reinterpret_cast<const int4*>(ids);
  int4* pos4 = reinterpret_cast<int4*>(rank_of_pair);
  auto rank_of = [&](int e) { return (e >= 0 && e < E) ? static_cast<int>(atomicAdd(&cnt[e], 1u)) : -1; };
  for (int q0 = tid; q0 < n4; q0 += 8 * kRouteThreads) {
    int4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = q0 + u * kRouteThreads;
      v[u] = q < n4 ? __ldg(ids4 + q) : make_int4(-1, -1, -1, -1);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = q0 + u * kRouteThreads;
      if (q < n4) pos4[q] = make_int4(rank_of(v[u].x), rank_of(v[u].y), rank_of(v[u].z), rank_of(v[u].w));
    }
  }
  for (int i = 4 * n4 + tid; i < n_pairs; i += kRouteThreads) rank_of_pair[i] = rank_of(__ldg(ids + i));
  __syncthreads();
  // exclusive scans over the experts (one per thread, E <= 1024) of the
  // padded segment sizes and of the token tiles
  const uint32_t c = tid < E ? cnt[tid] : 0u;
  const uint32_t tiles = (c + 127u) / 128u, pad = tiles * 128u;
  uint32_t ip = pad, it = tiles;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t a = __shfl_up_sync(0xFFFFFFFFu, ip, d), b = __shfl_up_sync(0xFFFFFFFFu, it, d);
    if (lane >= d) { ip += a; it += b; }
  }
  if (lane == 31) { wpad[warp] = ip; wtile[warp] = it; }
  __syncthreads();
  if (warp == 0) {
    uint32_t sp = wpad[lane], st = wtile[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t a = __shfl_up_sync(0xFFFFFFFFu, sp, d), b = __shfl_up_sync(0xFFFFFFFFu, st, d);
      if (lane >= d) { sp += a; st += b; }
    }
    wpad[lane] = sp;
    wtile[lane] = st;
  }
  __syncthreads();
  const uint32_t base_p = (warp ? wpad[warp - 1] : 0u) + ip - pad;
  const uint32_t base_t = (warp ? wtile[warp - 1] : 0u) + it - tiles;
  if (tid < E) {
    seg_start[tid] = base_p;
    seg_count[tid] = c;
    for (uint32_t u = 0; u < tiles; ++u) units[base_t + u] = (static_cast<uint32_t>(tid) << 16) | u;
  }
  if (tid == 0) {
    ctl[0] = wtile[31];
    ctl[1] = wpad[31];
  }
}

// ------------------------------------------------------- quantize-scatter
// x quantized once per 16-element block pair (the standalone quantizer's
// arithmetic: identical codes and scale bytes) and stored into each of the
// token's k segment rows, seg_start[ids[t, j]] + rank: codes at [row, D/2],
// scale bytes in the tile layout; the thread of the row's first blocks also
// records the row's pair (row_of).  Rows of padding keep whatever they held
// (zero or an earlier call's finite codes; row_of is never read there): they
// only feed accumulator columns that are never stored.  A pair whose id is
// outside [0, E) gets a zero output row (each thread zeroes a slice).
template <bool kBF16>
__global__ void __launch_bounds__(256)
moe_quantize_scatter_kernel(const void* __restrict__ x, int T, int D, int k, const float* __restrict__ qrec,
                            const int32_t* __restrict__ ids, const int32_t* __restrict__ rank_of_pair,
                            const uint32_t* __restrict__ seg_start, int32_t* __restrict__ row_of, uint8_t* __restrict__ pc,
                            uint8_t* __restrict__ psf, void* __restrict__ y, int N, int y_bf16) {
  __shared__ float s_rcp[128];                 // RN(1 / dec(b)) for scale bytes b
  if (threadIdx.x < 128) {
    const uint32_t b = threadIdx.x;
    s_rcp[b] = (b >= 1 && b <= 126) ? __frcp_rn(e4m3_value(b)) : 0.0f;
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int KB = D / kBlock;
  const int pairs_per_row = KB / 2;
  const int64_t n_thr = static_cast<int64_t>(T) * pairs_per_row;
  QuantScale qs;
  qs.gsa = __ldg(qrec);
  qs.rgsa = __ldg(qrec + 1);
  qs.mode = __float_as_int(__ldg(qrec + 2));
  for (int64_t g0 = static_cast<int64_t>(blockIdx.x) * blockDim.x; g0 < n_thr;
       g0 += static_cast<int64_t>(gridDim.x) * blockDim.x) {   // block-uniform trip count
    const int64_t g = g0 + threadIdx.x;
    const bool live = g < n_thr;
    const int64_t t = live ? g / pairs_per_row : 0;
    const int c = live ? 2 * static_cast<int>(g - t * pairs_per_row) : 0;    // first block of the pair
    uint4 q = make_uint4(0u, 0u, 0u, 0u);
    uint32_t b0 = 0, b1 = 0;
    if (live) {
      Block16 blk;
      const size_t e0 = static_cast<size_t>(t) * D + static_cast<size_t>(c) * kBlock;
      load_block16<kBF16>(x, e0, blk);
      b0 = quant_block16_bracket(blk, qs, q.x, q.y, s_rcp);
      load_block16<kBF16>(x, e0 + kBlock, blk);
      b1 = quant_block16_bracket(blk, qs, q.z, q.w, s_rcp);
    }
    // blocks 4c'..4c'+3 of a row are 4 consecutive bytes of one tile line:
    // the even lane of each pair of lanes writes them (KB % 4 == 0, so both
    // lanes hold the same row)
    const uint32_t o = __shfl_down_sync(0xFFFFFFFFu, b0 | (b1 << 8), 1);
    if (live) {
      // the k destination rows first: all id and rank loads in flight at once
      int32_t rk[kMaxKmax], ex[kMaxKmax];
#pragma unroll
      for (int j = 0; j < kMaxKmax; ++j) {
        rk[j] = j < k ? __ldg(rank_of_pair + t * k + j) : -1;
        ex[j] = j < k ? __ldg(ids + t * k + j) : 0;
      }
      int64_t row[kMaxKmax];
#pragma unroll
      for (int j = 0; j < kMaxKmax; ++j) row[j] = rk[j] >= 0 ? static_cast<int64_t>(__ldg(seg_start + ex[j])) + rk[j] : -1;
#pragma unroll
      for (int j = 0; j < kMaxKmax; ++j) {
        if (j >= k) break;
        const int64_t pair = t * k + j, p = row[j];
        if (p < 0) {
          // an id outside [0, E): the pair's output row is zero
          for (int n = c * 8; n < N; n += KB * 8) {      // slices of 16 outputs, KB / 2 threads per row
            for (int u = 0; u < 16 && n + u < N; ++u) {
              if (y_bf16) reinterpret_cast<uint16_t*>(y)[pair * N + n + u] = 0;
              else reinterpret_cast<float*>(y)[pair * N + n + u] = 0.0f;
            }
          }
          continue;
        }
        *reinterpret_cast<uint4*>(pc + static_cast<size_t>(p) * (D / 2) + static_cast<size_t>(c) * 8) = q;
        if ((c & 3) == 0)
          *reinterpret_cast<uint32_t*>(psf + sf_tile_offset(p, c, KB)) = b0 | (b1 << 8) | (o << 16);
        if (c == 0) row_of[p] = static_cast<int32_t>(pair);
      }
    }
  }
}

// ------------------------------------------------------------ grouped GEMM
struct MoeParams {
  CUtensorMap tmap_w;          // expert weights [E * N, D/2], box 128 x 128, 128-byte swizzle
  CUtensorMap tmap_x;          // segment rows [P, D/2], box 128 x 128, 128-byte swizzle
  const uint8_t* sfw;          // expert weight scales, tile layout over E * N rows
  const uint8_t* sfx;          // segment row scales, tile layout
  const float* x_gsa;
  const float* w_gsa;          // [E]
  const uint32_t* seg_start;
  const uint32_t* seg_count;
  const uint32_t* units;
  const uint32_t* ctl;
  const int32_t* row_of;
  int D, N, n_nt;              // n_nt = N / 128 weight tiles per expert
  void* y;                     // [T * k, N]
  int y_bf16;
  uint32_t* status;
};

struct Unit {
  int e, row0, valid, wrow0;   // expert, first segment row, rows of the unit, first weight row
};

__device__ __forceinline__ Unit unit_of(const MoeParams& p, int w) {
  const int ui = w / p.n_nt, i = w - ui * p.n_nt;
  const uint32_t ue = __ldcg(p.units + ui);
  Unit u;
  u.e = static_cast<int>(ue >> 16);
  const int tt = static_cast<int>(ue & 0xFFFFu);
  u.row0 = static_cast<int>(__ldcg(p.seg_start + u.e)) + tt * 128;
  u.valid = min(128, static_cast<int>(__ldcg(p.seg_count + u.e)) - tt * 128);
  u.wrow0 = u.e * p.N + i * 128;
  return u;
}

__global__ void __launch_bounds__(kMThreads, 1)
moe_gemm_kernel(const __grid_constant__ MoeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int32_t* s_rows = reinterpret_cast<int32_t*>(smem + kMStages * kMStage);            // [128]
  uint64_t* full = reinterpret_cast<uint64_t*>(s_rows + 128);
  uint64_t* empty = full + kMStages;
  uint64_t* acc_full = empty + kMStages;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  uint32_t filled_mask = 0, fill_bits = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = p.D / kBlock;
  const int k_stages = (KB / 4 + 3) / 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMStages; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(acc_full + b, 1); mbar_init(acc_empty + b, kMEpi); }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&p.tmap_w);
    tma_prefetch_map(&p.tmap_x);
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const uint64_t deadline = globaltimer_ns() + 1000000000ull;
  const int n_work = static_cast<int>(__ldcg(p.ctl)) * p.n_nt;
  const int n_mine = n_work > static_cast<int>(blockIdx.x)
                         ? (n_work - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                               static_cast<int>(gridDim.x)
                         : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = 0; it < n_mine && ok; ++it) {
      const Unit u = unit_of(p, blockIdx.x + it * gridDim.x);
      for (int ks = 0; ks < k_stages; ++ks) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty + stage, phase ^ 1u, deadline, abort_flag))) {
          ok = false;
          break;
        }
        const int nkk = min(4, KB / 4 - 4 * ks);
        uint8_t* a = smem + stage * kMStage;
        uint8_t* b = a + kMTile;
        uint8_t* sa = b + kMTile;
        uint8_t* sb = sa + kMSlab;
        if (elect_one()) {
          mbar_arrive_expect_tx(full + stage, 2u * kMTile + 2u * 512u * nkk);
          tma_load_2d(a, &p.tmap_w, ks * 128, u.wrow0, full + stage);
          tma_load_2d(b, &p.tmap_x, ks * 128, u.row0, full + stage);
          bulk_load(sa, p.sfw + (static_cast<size_t>(u.wrow0 / 128) * (KB / 4) + 4 * ks) * 512, 512u * nkk,
                    full + stage);
          bulk_load(sb, p.sfx + (static_cast<size_t>(u.row0 / 128) * (KB / 4) + 4 * ks) * 512, 512u * nkk,
                    full + stage);
        }
        __syncwarp();
        filled_mask |= 1u << stage;
        fill_bits = (fill_bits & ~(1u << stage)) | (phase << stage);
        if (++stage == kMStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      report_timeout(p.status);
      *abort_flag = 1;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t kIdesc = idesc_mxf4nvf4(128, 128);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = 0; it < n_mine && ok; ++it) {
      const int buf = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(acc_empty + buf, acc_phase ^ 1u, deadline, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + buf * 128;
      for (int ks = 0; ks < k_stages; ++ks) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(full + stage, phase, deadline, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int nkk = min(4, KB / 4 - 4 * ks);
        const uint8_t* a = smem + stage * kMStage;
        const uint8_t* b = a + kMTile;
        const uint8_t* sa = b + kMTile;
        const uint8_t* sb = sa + kMSlab;
        const uint32_t sfa_t = tmem + 256 + stage * 32;
        const uint32_t sfb_t = sfa_t + 16;
        if (elect_one()) {
          for (int kk = 0; kk < nkk; ++kk) {
            tc_copy_scales(sfa_t + 4 * kk, desc_scale_tile(smem_u32(sa + 512 * kk)));
            tc_copy_scales(sfb_t + 4 * kk, desc_scale_tile(smem_u32(sb + 512 * kk)));
          }
          for (int kk = 0; kk < nkk; ++kk)
            tc_mma_nvf4(d_tmem, desc_kmajor_sw128(smem_u32(a + 32 * kk)), desc_kmajor_sw128(smem_u32(b + 32 * kk)),
                        kIdesc, sfa_t + 4 * kk, sfb_t + 4 * kk, (ks | kk) != 0);
          tc_commit(empty + stage);
        }
        __syncwarp();
        if (++stage == kMStages) { stage = 0; phase ^= 1u; }
      }
      if (ok && elect_one()) tc_commit(acc_full + buf);
      __syncwarp();
    }
    if (!ok && lane == 0) {
      report_timeout(p.status);
      *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warp pair (quarter q, half h): weight rows 32q.. of the tile, token
    // columns 64h..64h+63; consecutive lanes hold consecutive outputs n, so
    // every y store is coalesced along the row
    const int et = threadIdx.x - 64;
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int wrow = quarter * 32 + lane;
    const float x_gsa = __ldg(p.x_gsa);
    bool ok = true;
    for (int it = 0; it < n_mine; ++it) {
      const int buf = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const Unit u = unit_of(p, blockIdx.x + it * gridDim.x);
      const float gscale = __fmul_rn(x_gsa, __ldg(p.w_gsa + u.e));
      // the unit's output rows (the previous unit's readers are done: the
      // barrier at the end of the loop)
      if (et < 128) s_rows[et] = et < u.valid ? __ldcg(p.row_of + u.row0 + et) : -1;
      const bool got = bar_and(1, kMEpi, mbar_wait(acc_full + buf, acc_phase, deadline, abort_flag));
      if (!got) { ok = false; break; }
      tc_fence_after();
      const int n = (u.wrow0 - u.e * p.N) + wrow;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        float v[32];
        const int t0 = half * 64 + c * 32;
        tmem_load32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * 128 + t0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int row = s_rows[t0 + i];
          if (row >= 0) {
            const float val = __fmul_rn(v[i], gscale);
            const size_t o = static_cast<size_t>(row) * p.N + n;
            if (p.y_bf16) {
              const __nv_bfloat16 h = __float2bfloat16_rn(val);
              reinterpret_cast<__nv_bfloat16*>(p.y)[o] = h;
            } else {
              reinterpret_cast<float*>(p.y)[o] = val;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty + buf);
      asm volatile("bar.sync 2, 256;" ::: "memory");       // s_rows is free again
    }
    if (!ok) {
      report_timeout(p.status);
      *abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort_flag && threadIdx.x == 0) {
    const uint64_t drain = globaltimer_ns() + 1000000000ull;
    for (int s = 0; s < kMStages; ++s) {
      if (!((filled_mask >> s) & 1u)) continue;
      while (!mbar_try_wait(full + s, (fill_bits >> s) & 1u))
        if (globaltimer_ns() > drain) break;
    }
  }
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- combine
// out[t, n] = sum_j w[t, j] * y[t, j, n], j in order (fused multiply-adds),
// four outputs per thread.
template <bool kBF16>
__global__ void __launch_bounds__(256)
moe_combine_kernel(const void* __restrict__ y, int64_t T, int k, int N, const float* __restrict__ w,
                   float* __restrict__ out) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int nq = N / 4;
  const int64_t total = T * nq;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = g / nq;
    const int n = static_cast<int>(g - t * nq) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float wt = __ldg(w + t * k + j);
      const size_t o = (static_cast<size_t>(t) * k + j) * N + n;
      float4 v;
      if (kBF16) {
        const uint2 b = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(y) + o));
        v = make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u), __uint_as_float(b.y << 16),
                        __uint_as_float(b.y & 0xFFFF0000u));
      } else {
        v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(y) + o));
      }
      acc.x = __fmaf_rn(wt, v.x, acc.x);
      acc.y = __fmaf_rn(wt, v.y, acc.y);
      acc.z = __fmaf_rn(wt, v.z, acc.z);
      acc.w = __fmaf_rn(wt, v.w, acc.w);
    }
    *reinterpret_cast<float4*>(out + t * N + n) = acc;
  }
}

size_t a256(size_t v) { return (v + 255) / 256 * 256; }

// Workspace of a grouped GEMM call: the quantize layout (control words, amax
// partials, x's quantizer record) then the routing tables and the rows.
struct MoeWs {
  size_t ctl, seg_start, seg_count, units, pos_of, row_of, pc, psf, total;
  int64_t rows_max;            // rows of all segments at most (128-padded)
};

MoeWs moe_ws_layout(int64_t T, int64_t D, int64_t E, int k) {
  MoeWs L;
  const int64_t pairs = T * k;
  L.rows_max = (pairs + E * 127 + 127) / 128 * 128;
  const size_t q = quantize_ws_layout(T, D).total;
  L.ctl = a256(q);
  L.seg_start = L.ctl + 256;
  L.seg_count = a256(L.seg_start + E * 4);
  L.units = a256(L.seg_count + E * 4);
  L.pos_of = a256(L.units + ((pairs + 127) / 128 + E) * 4);
  L.row_of = a256(L.pos_of + pairs * 4);
  L.pc = a256(L.row_of + L.rows_max * 4);
  L.psf = a256(L.pc + L.rows_max * (D / 2));
  L.total = a256(L.psf + L.rows_max * (D / 16));
  return L;
}

bool encode_rows(CUtensorMap* map, const uint8_t* ptr, int64_t rows, int64_t D) {
  return encode_codes(map, ptr, rows, D, 128);
}

}  // namespace

}  // namespace nvr

using namespace nvr;

extern "C" size_t nvfp4_moe_gemm_workspace_size(int64_t T_max, int64_t D, int64_t n_experts, int k) {
  if (T_max < 0 || D <= 0 || D % 64 != 0 || n_experts < 1 || n_experts > kMoeMaxExperts || k < 1 || k > kMaxKmax)
    return 0;
  return moe_ws_layout(T_max, D, n_experts, k).total;
}

extern "C" nvr_status nvfp4_moe_gemm(const void* x, nvr_dtype dt, int64_t T, int64_t D, const int32_t* ids, int k,
                                     int64_t n_experts, const uint8_t* W_fp4, const uint8_t* W_scales,
                                     const float* w_gsa, int64_t N, void* y, nvr_dtype y_dt, void* workspace,
                                     size_t ws_bytes, nvr_stream_t stream) {
  if (!x || !ids || !W_fp4 || !W_scales || !w_gsa || !y || !workspace) return NVR_ERR_INVALID_ARG;
  if (T < 0 || D <= 0 || D % 64 != 0 || D > (1 << 24) || k < 1 || k > kMaxKmax) return NVR_ERR_INVALID_ARG;
  if (n_experts < 1 || n_experts > kMoeMaxExperts || N < 128 || N % 128 != 0) return NVR_ERR_INVALID_ARG;
  if ((dt != NVR_BF16 && dt != NVR_F32) || (y_dt != NVR_BF16 && y_dt != NVR_F32)) return NVR_ERR_INVALID_ARG;
  if (n_experts * N > (int64_t(1) << 31) || T * k > (int64_t(1) << 28)) return NVR_ERR_UNSUPPORTED;
  const uintptr_t a16 = 15u;
  if ((reinterpret_cast<uintptr_t>(x) & a16) || (reinterpret_cast<uintptr_t>(W_fp4) & a16) ||
      (reinterpret_cast<uintptr_t>(W_scales) & a16) || (reinterpret_cast<uintptr_t>(y) & a16) ||
      (reinterpret_cast<uintptr_t>(ids) & 15u) || (reinterpret_cast<uintptr_t>(w_gsa) & 3u) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return NVR_ERR_ALIGNMENT;
  const MoeWs L = moe_ws_layout(T, D, n_experts, k);
  if (ws_bytes < L.total) return NVR_ERR_WORKSPACE;
  if (L.rows_max * (D / 32) >= (int64_t(1) << 31)) return NVR_ERR_UNSUPPORTED;
  if (T == 0) return NVR_OK;
  const int sms = device_sm_count();
  if (sms <= 0) return NVR_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  const WsLayout Q = quantize_ws_layout(T, D);
  float* x_gsa = reinterpret_cast<float*>(w + Q.scalars);
  float* qrec = x_gsa + 4;
  uint32_t* status = reinterpret_cast<uint32_t*>(w + kWsStatus);
  const bool bf16 = dt == NVR_BF16;
  cudaError_t e = launch_amax_bulk(x, bf16, T * D, reinterpret_cast<uint32_t*>(w + Q.amax_partials),
                                   reinterpret_cast<uint32_t*>(w + kWsAmaxTicket), x_gsa, qrec, status, sms, s);
  if (e != cudaSuccess) return cuda_status(e);

  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  uint32_t* ctl = reinterpret_cast<uint32_t*>(w + L.ctl);
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kRouteThreads);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, moe_route_kernel, ids, static_cast<int>(T * k), static_cast<int>(n_experts),
                           reinterpret_cast<int32_t*>(w + L.pos_of), reinterpret_cast<uint32_t*>(w + L.seg_start),
                           reinterpret_cast<uint32_t*>(w + L.seg_count), reinterpret_cast<uint32_t*>(w + L.units), ctl);
    if (e != cudaSuccess) return cuda_status(e);
  }
  {
    const int64_t n_thr = T * (D / kBlock / 2);
    int64_t grid = (n_thr + 255) / 256;
    if (grid > static_cast<int64_t>(sms) * 32) grid = static_cast<int64_t>(sms) * 32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    const int32_t* rk = reinterpret_cast<const int32_t*>(w + L.pos_of);
    const uint32_t* ss = reinterpret_cast<const uint32_t*>(w + L.seg_start);
    int32_t* ro = reinterpret_cast<int32_t*>(w + L.row_of);
    const int yb = y_dt == NVR_BF16 ? 1 : 0, n32 = static_cast<int>(N), t32 = static_cast<int>(T),
              d32 = static_cast<int>(D);
    const float* qr = qrec;
    e = bf16 ? cudaLaunchKernelEx(&cfg, moe_quantize_scatter_kernel<true>, x, t32, d32, k, qr, ids, rk, ss, ro,
                                  w + L.pc, w + L.psf, y, n32, yb)
             : cudaLaunchKernelEx(&cfg, moe_quantize_scatter_kernel<false>, x, t32, d32, k, qr, ids, rk, ss, ro,
                                  w + L.pc, w + L.psf, y, n32, yb);
    if (e != cudaSuccess) return cuda_status(e);
  }
  MoeParams p;
  if (!encode_rows(&p.tmap_w, W_fp4, n_experts * N, D)) return NVR_ERR_UNSUPPORTED;
  if (!encode_rows(&p.tmap_x, w + L.pc, L.rows_max, D)) return NVR_ERR_UNSUPPORTED;
  p.sfw = W_scales; p.sfx = w + L.psf; p.x_gsa = x_gsa; p.w_gsa = w_gsa;
  p.seg_start = reinterpret_cast<const uint32_t*>(w + L.seg_start);
  p.seg_count = reinterpret_cast<const uint32_t*>(w + L.seg_count);
  p.units = reinterpret_cast<const uint32_t*>(w + L.units);
  p.ctl = ctl;
  p.row_of = reinterpret_cast<const int32_t*>(w + L.row_of);
  p.D = static_cast<int>(D); p.N = static_cast<int>(N); p.n_nt = static_cast<int>(N / 128);
  p.y = y; p.y_bf16 = y_dt == NVR_BF16 ? 1 : 0; p.status = status;
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVR_ERR_CUDA;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(moe_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMSmem);
    if (e != cudaSuccess) return cuda_status(e);
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms));
  cfg.blockDim = dim3(kMThreads);
  cfg.dynamicSmemBytes = kMSmem;
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, moe_gemm_kernel, p));
}

extern "C" nvr_status nvfp4_moe_combine(const void* y, nvr_dtype y_dt, int64_t T, int k, int64_t N, const float* w,
                                        float* out, nvr_stream_t stream) {
  if (T < 0 || k < 1 || k > kMaxKmax || N < 4 || N % 4 != 0 || N > (1 << 28)) return NVR_ERR_INVALID_ARG;
  if (y_dt != NVR_BF16 && y_dt != NVR_F32) return NVR_ERR_INVALID_ARG;
  if (T > 0 && (!y || !w || !out)) return NVR_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(y) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u) ||
      (reinterpret_cast<uintptr_t>(w) & 3u))
    return NVR_ERR_ALIGNMENT;
  if (T == 0) return NVR_OK;
  const int sms = device_sm_count();
  if (sms <= 0) return NVR_ERR_CUDA;
  const int64_t total = T * (N / 4);
  int64_t grid = (total + 255) / 256;
  if (grid > static_cast<int64_t>(sms) * 16) grid = static_cast<int64_t>(sms) * 16;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(256);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  const int n32 = static_cast<int>(N);
  return cuda_status(y_dt == NVR_BF16
                         ? cudaLaunchKernelEx(&cfg, moe_combine_kernel<true>, y, T, k, n32, w, out)
                         : cudaLaunchKernelEx(&cfg, moe_combine_kernel<false>, y, T, k, n32, w, out));
}
