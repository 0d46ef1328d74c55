// gemm_topk.cu -- block-scaled NVFP4 gate GEMM on the 5th-generation tensor
// cores with the router epilogue fused on the accumulator (sm_103a).
//
// Source: "nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py"
// (NVFP4 gate GEMM on Blackwell tensor cores; the single-kernel block-scaled
// GEMM + fused router epilogue of the fused dispatch section) and
// "commit e0f60b9: dsv4/kernels/router/__init__.py" (activation_topk's six
// steps; the row-level top-k that spans N-subtiles, which is not a
// per-element epilogue).
//
// Tiling.  A CTA owns one 128-token M tile and a strided subset of the
// 128-expert N tiles ("split" s of n_splits handles N tiles s, s + n_splits,
// ...).  For each N tile the K loop runs in stages of 256 elements (128 bytes
// of packed codes per row, one 128-byte swizzle atom):
//   warp 0 (one thread)  TMA: the x tile and the W tile (128 x 128 bytes each,
//                        128-byte swizzle) and the two 2 KB scale slabs
//                        (4 tiles of 128 rows x 4 scale columns) per stage,
//                        into a 6-deep shared-memory ring;
//   warp 1 (one thread)  copies each stage's scales to tensor memory
//                        (tcgen05.cp) and issues four
//                        tcgen05.mma.kind::mxf4nvf4.block_scale (M=128, N=128,
//                        K=64) into one of two fp32 accumulators in tensor
//                        memory; tcgen05.commit frees the stage / publishes
//                        the accumulator;
//   warps 2-5            epilogue: each thread owns one token row (one tensor
//                        memory lane), reads its 128 logits with tcgen05.ld,
//                        applies gsa_x * gsa_w, sigmoid, + bias and keeps a
//                        sorted top-k in registers across all of the CTA's N
//                        tiles, while the MMA warp fills the other
//                        accumulator.
// Logits never leave the chip.  When N is split across CTAs, each CTA writes
// its per-row top-k list to the workspace and the last CTA of the M tile
// (atomic ticket, no waiting) merges the lists in split order, renormalises
// and writes ids and weights.
//
// Tensor memory (512 columns): accumulators at columns 0 and 128; the scale
// tiles of ring stage s at 256 + 32 s (A: 16 columns, B: 16 columns).
#include "nvr_internal.h"
#include "nvr_tcgen05.cuh"

namespace nvr {

constexpr int kStages = 5;
constexpr int kTileBytes = 128 * 128;              // 128 rows x 128 bytes
constexpr int kSfSlab = 4 * 512;                   // 4 scale tiles
constexpr int kStageBytes = 2 * kTileBytes + 2 * kSfSlab;
constexpr int kEpiChunk = 32;                       // columns per tensor-memory load
constexpr int kEpiBytes = kEpiChunk * 256 * 4;      // logits of one chunk, every epilogue thread
constexpr int kGemmSmem = kStages * kStageBytes + 1024 /*barriers*/ + 1024 /*bias*/ + kEpiBytes +
                          1024 /*align*/;
constexpr int kGemmThreads = 320;                  // producer, MMA, 8 epilogue warps
constexpr uint32_t kIdesc = idesc_mxf4nvf4(128, 128);

struct GemmParams {
  CUtensorMap tmap_a;          // x codes [T, D/2] uint8
  CUtensorMap tmap_b;          // W codes [N, D/2] uint8
  const uint8_t* sfa;          // x scales, tile layout
  const uint8_t* sfb;          // W scales, tile layout
  const float* x_gsa;
  const float* w_gsa;
  const float* bias;           // [N] or null
  int T, N, D, k;
  int raw, n_splits, n_tiles;
  float routed_scaling;
  int32_t* out_ids;
  float* out_w;
  void* logits;                // logits mode: write [T, N] logits (fp32, or bf16) instead of the top-k
  int logits_bf16;
  float4* partials;            // [m_tiles * n_splits][128][KMAX]
  uint32_t* tickets;           // [m_tiles]
  uint32_t* status;
  int test_stall;              // test hook: the MMA issuer issues nothing
};

template <int KMAX>
__device__ __forceinline__ void write_final(const TopK<KMAX>& tk, const GemmParams& p, int64_t token) {
  int32_t* ids = p.out_ids + token * p.k;
  float* w = p.out_w + token * p.k;
  if (p.raw) {
#pragma unroll
    for (int i = 0; i < KMAX; ++i)
      if (i < p.k) { ids[i] = tk.id[i]; w[i] = tk.sc[i]; }
    return;
  }
  float sum = 0.0f;
#pragma unroll
  for (int i = 0; i < KMAX; ++i)
    if (i < p.k) sum = __fadd_rn(sum, tk.sc[i]);
#pragma unroll
  for (int i = 0; i < KMAX; ++i)
    if (i < p.k) {
      ids[i] = tk.id[i];
      w[i] = sum > 0.0f ? __fdiv_rn(__fmul_rn(p.routed_scaling, tk.sc[i]), sum) : 0.0f;
    }
}

template <int KMAX>
__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_topk_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* last_flag = abort_flag + 1;
  volatile int* epi_abort = abort_flag + 2;     // the epilogue's agreed view of abort_flag
  float* s_bias = reinterpret_cast<float*>(smem + kStages * kStageBytes + 1024);   // [2][128]
  float* s_lg = s_bias + 2 * 128;                   // [kEpiChunk][256] logits, column per thread

  // producer thread: which ring stages were filled, and the parity of each
  // stage's latest fill (bit s)
  uint32_t filled_mask = 0, fill_bits = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x / p.n_splits;
  const int split = blockIdx.x - m_tile * p.n_splits;
  const int n_mine = (p.n_tiles - split + p.n_splits - 1) / p.n_splits;
  const int KB = p.D / kBlock;
  const int k_stages = (KB / 4 + 3) / 4;          // 4 scale tiles (K = 256) per stage

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(acc_full + b, 1); mbar_init(acc_empty + b, 256); }
    *abort_flag = 0;
    *last_flag = 0;
    *epi_abort = 0;
    fence_mbar_init();
    tma_prefetch_map(&p.tmap_a);
    tma_prefetch_map(&p.tmap_b);
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // the quantize kernel before us (programmatic launch) must have finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint64_t deadline = globaltimer_ns() + 1000000000ull;   // 1 s

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (uniform control flow); one elected lane
    // issues the copies.
    {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0; it < n_mine && ok; ++it) {
        const int j = split + it * p.n_splits;
        for (int ks = 0; ks < k_stages; ++ks) {
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty + stage, phase ^ 1u, deadline, abort_flag))) {
            ok = false;
            break;
          }
          const int nkk = min(4, KB / 4 - 4 * ks);
          uint8_t* a = smem + stage * kStageBytes;
          uint8_t* b = a + kTileBytes;
          uint8_t* sa = b + kTileBytes;
          uint8_t* sb = sa + kSfSlab;
          if (elect_one()) {
            mbar_arrive_expect_tx(full + stage, 2u * kTileBytes + 2u * 512u * nkk);
            tma_load_2d(a, &p.tmap_a, ks * 128, m_tile * 128, full + stage);
            tma_load_2d(b, &p.tmap_b, ks * 128, j * 128, full + stage);
            bulk_load(sa, p.sfa + (static_cast<size_t>(m_tile) * (KB / 4) + 4 * ks) * 512, 512u * nkk,
                      full + stage);
            bulk_load(sb, p.sfb + (static_cast<size_t>(j) * (KB / 4) + 4 * ks) * 512, 512u * nkk,
                      full + stage);
          }
          __syncwarp();
          filled_mask |= 1u << stage;
          fill_bits = (fill_bits & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok && lane == 0) {
        report_timeout(p.status);
        *abort_flag = 1;
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs the loop; one elected lane issues the tensor-core
    // work and its commits (a commit tracks the issuing thread's operations).
    if (!p.test_stall) {
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
          const uint8_t* a = smem + stage * kStageBytes;
          const uint8_t* b = a + kTileBytes;
          const uint8_t* sa = b + kTileBytes;
          const uint8_t* sb = sa + kSfSlab;
          const uint32_t sfa_t = tmem + 256 + stage * 32;
          const uint32_t sfb_t = sfa_t + 16;
          if (elect_one()) {
            for (int kk = 0; kk < nkk; ++kk) {
              tc_copy_scales(sfa_t + 4 * kk, desc_scale_tile(smem_u32(sa + 512 * kk)));
              tc_copy_scales(sfb_t + 4 * kk, desc_scale_tile(smem_u32(sb + 512 * kk)));
            }
            for (int kk = 0; kk < nkk; ++kk) {
              tc_mma_nvf4(d_tmem, desc_kmajor_sw128(smem_u32(a + 32 * kk)),
                          desc_kmajor_sw128(smem_u32(b + 32 * kk)), kIdesc, sfa_t + 4 * kk,
                          sfb_t + 4 * kk, (ks | kk) != 0);
            }
            tc_commit(empty + stage);
          }
          __syncwarp();
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (ok && elect_one()) tc_commit(acc_full + buf);
        __syncwarp();
      }
      if (!ok && lane == 0) {
        report_timeout(p.status);
        *abort_flag = 1;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Eight warps: two per tensor-memory lane quarter, each owning half of
    // every tile's 128 columns for its 32 token rows, so two warps share each
    // scheduler and hide each other's latencies.
    const int etid = threadIdx.x - 64;             // 0..255
    const int half = etid >> 7;                    // columns [64*half, 64*half + 64) of a tile
    const int quarter = warp & 3;                  // tensor-memory lanes 32*quarter ..
    const int row = quarter * 32 + lane;
    const int64_t token = static_cast<int64_t>(m_tile) * 128 + row;
    const bool active = token < p.T;
    const float gscale = __fmul_rn(__ldg(p.x_gsa), __ldg(p.w_gsa));
    TopK<KMAX> tk;
    tk.init();
    bool ok = true;
    for (int it = 0; it < n_mine; ++it) {
      const int j = split + it * p.n_splits;
      const int buf = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      // Stage this N tile's bias in shared memory while the tile accumulates
      // (double-buffered by tile parity).
      float* tb = s_bias + buf * 128;
      if (etid < 128 && !p.raw && !p.logits) {
        const int n = j * 128 + etid;
        tb[etid] = (p.bias && n < p.N) ? __ldg(p.bias + n) : 0.0f;
      }
      // The epilogue warps agree on the outcome of the wait (one barrier that
      // also publishes the staged bias), so all of them leave the loop
      // together on a timeout and tcgen05.ld always runs warp-wide.
      const bool got = bar_and(1, 256, mbar_wait(acc_full + buf, acc_phase, deadline, abort_flag));
      if (!got) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int c = half * 2 + cc;               // 32-column chunk of the tile
        float v[32];
        tmem_load32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * 128 + c * 32, v);
        const int n0 = j * 128 + c * 32;
        if (p.logits) {
          // the warp's 32 rows x 32 columns through its own 4 KB of s_lg,
          // transposed (element (r, c) at r * 32 + (c ^ r): conflict-free both
          // ways), so that each store covers 32 consecutive columns of a row
          float* tr = s_lg + (etid >> 5) * 1024;
#pragma unroll
          for (int i = 0; i < 32; ++i) tr[lane * 32 + (i ^ lane)] = __fmul_rn(v[i], gscale);
          __syncwarp();
          const int64_t row0 = static_cast<int64_t>(m_tile) * 128 + quarter * 32;
          const int n = n0 + lane;
#pragma unroll 4
          for (int r = 0; r < 32; ++r) {
            const float l = tr[r * 32 + (lane ^ r)];
            if (row0 + r < p.T && n < p.N) {
              const size_t o = static_cast<size_t>(row0 + r) * p.N + n;
              if (p.logits_bf16) {
                const __nv_bfloat16 h = __float2bfloat16_rn(l);
                reinterpret_cast<__nv_bfloat16*>(p.logits)[o] = h;
              } else {
                reinterpret_cast<float*>(p.logits)[o] = l;
              }
            }
          }
          __syncwarp();
        } else {
          // Pass 1 (unrolled, branch-free): the exact key of every column of
          // the chunk; the logits go to this thread's column of s_lg.  A
          // keys-only sorted insertion (max/min only) of those keys into a copy
          // of the list's keys yields tau, the exact k-th largest key of the
          // list and the chunk together.  Only columns with key >= tau can
          // enter the list, so only they take the (costlier) exact insertion
          // with ids and scores: at most k of them plus exact ties.
          float sk[KMAX];
#pragma unroll
          for (int q = 0; q < KMAX; ++q) sk[q] = tk.key[q];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float l = __fmul_rn(v[i], gscale);
            s_lg[i * 256 + etid] = l;
            float key = l;
            if (!p.raw) {
              const float sc = sigmoid_f32(l);
              key = p.bias ? __fadd_rn(sc, tb[c * 32 + i]) : sc;
            }
            v[i] = (active && n0 + i < p.N) ? key : -INFINITY;
#pragma unroll
            for (int q = KMAX - 1; q > 0; --q) sk[q] = fmaxf(sk[q], fminf(sk[q - 1], v[i]));
            sk[0] = fmaxf(sk[0], v[i]);
          }
          const float tau = sk[KMAX - 1];
          uint32_t cand = 0;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            cand |= static_cast<uint32_t>(v[i] != -INFINITY && v[i] >= tau) << i;
          // Pass 2: the candidates enter the list.  With an 8-entry list, up
          // to 8 of them are gathered into fixed slots, sorted by a
          // 19-comparator network and merged with a bitonic merge (no
          // data-dependent control flow); any further candidates (exact ties
          // at tau) and lists of other sizes take the exact insertion.  Loops
          // run the same number of rounds in every lane of the warp (the
          // warp's largest candidate count), so the lanes stay converged.
          if constexpr (KMAX == 8) {
            float gk[8], gs[8];
            int gi[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              const bool has = cand != 0;
              const int i = has ? __ffs(cand) - 1 : 0;
              cand &= cand - 1;
              const float l = s_lg[i * 256 + etid];
              float key = l, sc = l;
              if (!p.raw) {
                sc = sigmoid_f32(l);
                key = p.bias ? __fadd_rn(sc, tb[c * 32 + i]) : sc;
              }
              gk[r] = has ? key : -INFINITY;
              gi[r] = has ? n0 + i : 0x7FFFFFFF;
              gs[r] = has ? sc : 0.0f;
            }
            if (__any_sync(0xFFFFFFFFu, gk[0] != -INFINITY)) {
              sort8(gk, gi, gs);
              tk.merge_sorted8(gk, gi, gs);
            }
          }
          const int rounds = __reduce_max_sync(0xFFFFFFFFu, static_cast<unsigned>(__popc(cand)));
#pragma unroll 1
          for (int r = 0; r < rounds; ++r) {
            const bool has = cand != 0;
            const int i = has ? __ffs(cand) - 1 : 0;
            cand &= cand - 1;
            const float l = s_lg[i * 256 + etid];
            float key = l, sc = l;
            if (!p.raw) {
              sc = sigmoid_f32(l);
              key = p.bias ? __fadd_rn(sc, tb[c * 32 + i]) : sc;
            }
            tk.push_if(key, n0 + i, sc, has);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty + buf);
    }
    if (!ok) {
      report_timeout(p.status);
      *abort_flag = 1;
    }
    // Agree on one abort decision before the named barriers below: every
    // epilogue thread has left its loop (bounded waits) and published its
    // failure; one thread snapshots the flag for all.
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (etid == 0) *epi_abort = *abort_flag;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (!*epi_abort && !p.logits) {
      // The two halves of each row merge: the second hands its list to the
      // first through shared memory.
      float* s_m = s_lg;                           // [KMAX][3][128]
      if (half == 1 && active) {
#pragma unroll
        for (int i = 0; i < KMAX; ++i) {
          s_m[(i * 3 + 0) * 128 + row] = tk.key[i];
          s_m[(i * 3 + 1) * 128 + row] = __int_as_float(tk.id[i]);
          s_m[(i * 3 + 2) * 128 + row] = tk.sc[i];
        }
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (half == 0) {
        if constexpr (KMAX == 8) {
          // both lists are sorted: one bitonic merge
          float bk[8], bs[8];
          int bi[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            bk[i] = s_m[(i * 3 + 0) * 128 + row];
            bi[i] = __float_as_int(s_m[(i * 3 + 1) * 128 + row]);
            bs[i] = s_m[(i * 3 + 2) * 128 + row];
          }
          if (active) tk.merge_sorted8(bk, bi, bs);
        } else {
          // warp-uniform loop; the half-1 list is sorted, so once no lane of
          // the warp has a qualifying entry left the rest cannot qualify either
#pragma unroll 1
          for (int i = 0; i < KMAX; ++i) {
            const float k2 = s_m[(i * 3 + 0) * 128 + row];
            const int i2 = __float_as_int(s_m[(i * 3 + 1) * 128 + row]);
            const bool q = active && topk_better(k2, i2, tk.key[KMAX - 1], tk.id[KMAX - 1]);
            if (!__any_sync(0xFFFFFFFFu, q)) break;
            tk.push_if(k2, i2, s_m[(i * 3 + 2) * 128 + row], q);
          }
        }
        asm volatile("bar.sync 2, 128;" ::: "memory");   // s_m is reused below
        if (p.n_splits == 1) {
          if (active) write_final<KMAX>(tk, p, token);
        } else {
          float4* dst = p.partials + (static_cast<size_t>(blockIdx.x) * 128 + row) * KMAX;
#pragma unroll
          for (int i = 0; i < KMAX; ++i) dst[i] = make_float4(tk.key[i], __int_as_float(tk.id[i]), tk.sc[i], 0.0f);
          __threadfence();
          asm volatile("bar.sync 2, 128;" ::: "memory");
          if (etid == 0) {
            const uint32_t t = atomicAdd(p.tickets + m_tile, 1u);
            *last_flag = (t == static_cast<uint32_t>(p.n_splits - 1)) ? 1 : 0;
          }
          asm volatile("bar.sync 2, 128;" ::: "memory");
          if (*last_flag) {
            __threadfence();
            TopK<KMAX> fin;
            fin.init();
            const float4* src = p.partials + static_cast<size_t>(m_tile) * p.n_splits * 128 * KMAX;
            // Every split's list is sorted, so a list is read only while its
            // next entry still beats the merged list's last one in some lane.
            // The heads of 8 lists are fetched together (staged in shared
            // memory) to overlap their latencies.  All loops are warp-uniform.
            float4* s_head = reinterpret_cast<float4*>(s_lg);     // [8][128]
            if constexpr (KMAX == 8) {
              // fold the sorted split lists in with bitonic merges, fetching
              // the next list while the current one merges
              float4 nxt[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) nxt[i] = __ldcg(src + static_cast<size_t>(row) * KMAX + i);
#pragma unroll 1
              for (int sp = 0; sp < p.n_splits; ++sp) {
                float bk[8], bs[8];
                int bi[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) { bk[i] = nxt[i].x; bi[i] = __float_as_int(nxt[i].y); bs[i] = nxt[i].z; }
                if (sp + 1 < p.n_splits) {
#pragma unroll
                  for (int i = 0; i < 8; ++i)
                    nxt[i] = __ldcg(src + (static_cast<size_t>(sp + 1) * 128 + row) * KMAX + i);
                }
                fin.merge_sorted8(bk, bi, bs);
              }
            }
            for (int s0 = 0; KMAX != 8 && s0 < p.n_splits; s0 += 8) {
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int sp = s0 + u;
                s_head[u * 128 + row] =
                    sp < p.n_splits ? __ldcg(src + (static_cast<size_t>(sp) * 128 + row) * KMAX)
                                    : make_float4(-INFINITY, __int_as_float(0x7FFFFFFF), 0.0f, 0.0f);
              }
#pragma unroll 1
              for (int u = 0; u < 8; ++u) {
                float4 h = s_head[u * 128 + row];
                const float4* e = src + (static_cast<size_t>(s0 + u < p.n_splits ? s0 + u : 0) * 128 + row) * KMAX;
                bool alive = active;
#pragma unroll 1
                for (int i = 0; i < KMAX; ++i) {
                  alive = alive && topk_better(h.x, __float_as_int(h.y), fin.key[KMAX - 1], fin.id[KMAX - 1]);
                  if (!__any_sync(0xFFFFFFFFu, alive)) break;
                  fin.push_if(h.x, __float_as_int(h.y), h.z, alive);
                  if (i + 1 < KMAX && alive) h = __ldcg(e + i + 1);
                }
              }
            }
            if (active) write_final<KMAX>(fin, p, token);
            if (etid == 0) p.tickets[m_tile] = 0u;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort_flag && threadIdx.x == 0) {
    // After an abort, copies issued by the producer may still be landing in
    // this CTA's shared memory: wait (bounded) for the latest fill of every
    // ring stage to complete before the CTA exits.
    const uint64_t drain = globaltimer_ns() + 1000000000ull;
    for (int s = 0; s < kStages; ++s) {
      if (!((filled_mask >> s) & 1u)) continue;
      while (!mbar_try_wait(full + s, (fill_bits >> s) & 1u)) {
        if (globaltimer_ns() > drain) break;
      }
    }
  }
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ launcher

template <int KMAX>
static cudaError_t launch_k(const GemmParams& p, int grid, cudaStream_t s) {
  static bool attr_set[kMaxDevices] = {};   // the attribute is per device and function
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(gemm_topk_kernel<KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = kGemmSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_topk_kernel<KMAX>, p);
}

static bool encode_codes_map(CUtensorMap* map, const uint8_t* ptr, int64_t rows, int64_t D) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D / 2), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D / 2)};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(ptr), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

GemmPlan plan_gemm(int64_t T, int64_t N, int num_sms) {
  GemmPlan g;
  g.m_tiles = static_cast<int>((T + 127) / 128);
  g.n_tiles = static_cast<int>((N + 127) / 128);
  int want = num_sms / (g.m_tiles > 0 ? g.m_tiles : 1);
  if (want < 1) want = 1;
  if (want > g.n_tiles) want = g.n_tiles;
  if (want > kMaxSplits) want = kMaxSplits;
  g.n_splits = want;
  return g;
}

nvr_status launch_gemm_topk(const uint8_t* x_codes, const uint8_t* x_sf, const float* x_gsa,
                            int64_t T, int64_t D, const uint8_t* W_codes, const uint8_t* W_sf,
                            const float* w_gsa, int64_t N, const float* bias, int k,
                            float routed_scaling, bool raw, int32_t* out_ids, float* out_w,
                            void* logits, bool logits_bf16, float4* partials, uint32_t* tickets,
                            uint32_t* status, const GemmPlan& g, bool test_stall, cudaStream_t s) {
  GemmParams p;
  if (!encode_codes_map(&p.tmap_a, x_codes, T, D)) return NVR_ERR_UNSUPPORTED;
  if (!encode_codes_map(&p.tmap_b, W_codes, N, D)) return NVR_ERR_UNSUPPORTED;
  p.sfa = x_sf; p.sfb = W_sf; p.x_gsa = x_gsa; p.w_gsa = w_gsa; p.bias = raw ? nullptr : bias;
  p.T = static_cast<int>(T); p.N = static_cast<int>(N); p.D = static_cast<int>(D); p.k = k;
  p.raw = raw ? 1 : 0; p.n_splits = g.n_splits; p.n_tiles = g.n_tiles;
  p.routed_scaling = routed_scaling;
  p.out_ids = out_ids; p.out_w = out_w; p.logits = logits; p.logits_bf16 = logits_bf16 ? 1 : 0;
  p.partials = partials; p.tickets = tickets; p.status = status;
  p.test_stall = test_stall ? 1 : 0;
  const int grid = g.m_tiles * g.n_splits;
  cudaError_t e;
  if (k <= 1) e = launch_k<1>(p, grid, s);
  else if (k <= 2) e = launch_k<2>(p, grid, s);
  else if (k <= 4) e = launch_k<4>(p, grid, s);
  else if (k <= 8) e = launch_k<8>(p, grid, s);
  else e = launch_k<16>(p, grid, s);
  return cuda_status(e);
}

}  // namespace nvr
