// gemm_stream.cu -- block-scaled NVFP4 GEMM for few tokens and many outputs
// (up to 128 tokens; wide router heads and the NVFP4 linear, e.g. an lm_head
// at decode batch sizes), streaming the weight through the tensor cores once
// (sm_103a).
//
// Source: "nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py"
// (NVFP4 block-scaled gate GEMM on Blackwell tensor cores, router epilogue
// fused on the accumulator; the top-k of a row spans N-subtiles) and
// "commit df05289: dsv4/layers/grouped_linear.py" (lm_head as an NVFP4 GEMM
// with a runtime activation scale, weight quantized at load time).
//
// Operand roles are swapped with respect to the token-tiled kernels: the MMA's
// M = 128 rows are 128 weight rows (outputs), its N = TN columns are the
// tokens (TN = 32, 64 or 128 >= T), so a tile wastes no tensor-core work on
// padding tokens and each weight byte is read from HBM exactly once.  CTA
// `split` of `n_splits` owns weight tiles split, split + n_splits, ... and
// runs, per tile, the K loop in stages of 256 elements:
//   warp 0     TMA producer: the weight tile (128 rows x 128 bytes, 128-byte
//              swizzle) with its 2 KB of scale atoms, and the token tile
//              (TN rows x 128 bytes) with its scale atoms, into a ring;
//   warp 1     MMA issuer: the stage's scale atoms into tensor memory
//              (tcgen05.cp), then four tcgen05.mma.kind::mxf4nvf4 (M = 128,
//              N = TN, K = 64) into one of several fp32 accumulators;
//   warps 2-9  epilogue, lane quarter q = warp % 4 (weight rows 32q..32q+31),
//              one weight row per thread, two warps per quarter taking half
//              of the TN token columns each: tcgen05.ld of the row's logits,
//              then either
//                - logits mode: out[t][n] = acc * gsa_x * gsa_w stored fp32 or
//                  bf16 -- consecutive lanes hold consecutive outputs n, so the
//                  stores are coalesced; or
//                - top-k mode: the tile goes through shared memory transposed
//                  (token-major); thread i takes token i % TN over TN / 2 of
//                  the tile's outputs and keeps a sorted (key, id, score) list
//                  in registers across all of the CTA's tiles (keys: the logit
//                  in RAW mode, else sigmoid(logit) + bias).
// Whenever a list's best entry changes it is published into the token's 32
// slots (slot id mod 32 keeps the best order-preserving (key, id) word, a
// 64-bit atomic max), and each CTA publishes its k best at the end; the k-th
// largest slot word is a lower bound of the token's global k-th best.  After its last tile a CTA merges its lists per
// token and appends only its entries at or above the bound to the token's
// candidates in the workspace, then takes a ticket; the last CTA (no
// waiting) selects each token's k best from its candidates -- a superset of
// them, a few per k once the bound has risen -- one warp per token (with at
// most 32 candidates each lane ranks one of them against the others),
// renormalises and writes ids and weights.
//
// Tensor memory (512 columns): kNacc accumulators of TN columns from column
// 0; the scale atoms of ring stage s at 256 + 32 s (weight: 16 columns,
// tokens: 16 columns) -- the tokens' atom holds 128 rows, of which the MMA
// reads the first TN.
#include "nvr_splitk.cuh"

namespace nvr {

namespace {

constexpr int kSThreads = 320;                 // producer, MMA, 8 epilogue warps
constexpr int kSEpi = 256;                     // epilogue threads
constexpr int kSWTile = 128 * 128;             // weight rows x 128 bytes of codes
constexpr int kSSfSlab = 4 * 512;              // 4 scale atoms (K = 256)

template <int TN> struct StreamCfg {
  static constexpr int kStages = TN == 128 ? 4 : (TN == 64 ? 5 : 6);
  static constexpr int kNacc = TN == 32 ? 4 : 2;
  static constexpr int kXTile = TN * 128;
  static constexpr int kStage = kSWTile + kSSfSlab + kXTile + kSSfSlab;
  static constexpr int kTrBytes = TN * 129 * 4;                 // transposed tile [TN][128 + 1] fp32
  static constexpr int kSmem = kStages * kStage + kTrBytes + 512 /*bias*/ + 1024 /*barriers*/ + 1024 /*align*/;
  static_assert(kStage % 1024 == 0, "1024-byte aligned stages");
  static_assert(kNacc * TN <= 256 && 256 + 32 * kStages <= 512, "tensor-memory budget");
  static_assert(kSmem <= 227 * 1024, "shared-memory budget");
};

struct StreamParams {
  CUtensorMap tmap_w;          // weight codes [N, D/2], box 128 x 128, 128-byte swizzle
  CUtensorMap tmap_x;          // token codes [T, D/2], box 128 x TN, 128-byte swizzle
  const uint8_t* sfw;          // weight scales, tile layout
  const uint8_t* sfx;          // token scales, tile layout (one 128-row atom per 4 K-blocks)
  const float* x_gsa;
  const float* w_gsa;
  const float* bias;           // [N] or null
  int T, N, D, k, raw, n_splits, n_tiles;
  float routed_scaling;
  int32_t* out_ids;
  float* out_w;
  void* out;                   // logits mode: [T, N] fp32 or bf16
  int out_bf16;
  // top-k mode with n_splits > 1 (workspace; every word is left at zero):
  float4* surv;                // [128][surv_stride] candidate (key, id, score, -) entries per token
  int surv_stride;             // n_splits * k
  uint32_t* ticket;            // CTAs done
  uint32_t* tok_count;         // [128] entries appended per token
  unsigned long long* tok_slots;   // [128][32] per token: the best (packed key, id) word published
                                   // by any CTA among the ids of each residue mod 32
  uint32_t* status;
  int test_stall;              // test hook: the MMA issuer issues nothing
};

__device__ __forceinline__ uint32_t bf16_rn_bits(float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  return static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&h));
}

template <int TN, int KMAX, bool kLogits>
__global__ void __launch_bounds__(kSThreads, 1)
gemm_stream_kernel(const __grid_constant__ StreamParams p) {
  using C = StreamCfg<TN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* s_tr = reinterpret_cast<float*>(smem + C::kStages * C::kStage);        // [TN][129]
  float* s_bias = s_tr + TN * 129;                                              // [128]
  uint64_t* full = reinterpret_cast<uint64_t*>(s_bias + 128);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + C::kNacc;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + C::kNacc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* last_flag = abort_flag + 1;
  volatile int* epi_abort = abort_flag + 2;

  uint32_t filled_mask = 0, fill_bits = 0;       // producer: ring stages with a fill in flight, their parity
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int n_mine = (p.n_tiles - split + p.n_splits - 1) / p.n_splits;
  const int KB = p.D / kBlock;
  const int k_stages = (KB / 4 + 3) / 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
    for (int b = 0; b < C::kNacc; ++b) { mbar_init(acc_full + b, 1); mbar_init(acc_empty + b, kSEpi); }
    *abort_flag = 0;
    *last_flag = 0;
    *epi_abort = 0;
    fence_mbar_init();
    tma_prefetch_map(&p.tmap_w);
    tma_prefetch_map(&p.tmap_x);
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // the quantize kernel before us (programmatic launch) must have finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const uint64_t deadline = globaltimer_ns() + 1000000000ull;   // 1 s

  if (warp == 0) {
    // ------------------------------------------------------------ producer
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
        uint8_t* a = smem + stage * C::kStage;
        uint8_t* sa = a + kSWTile;
        uint8_t* b = sa + kSSfSlab;
        uint8_t* sb = b + C::kXTile;
        if (elect_one()) {
          mbar_arrive_expect_tx(full + stage, static_cast<uint32_t>(kSWTile + C::kXTile + 2 * 512 * nkk));
          tma_load_2d(a, &p.tmap_w, ks * 128, j * 128, full + stage);
          tma_load_2d(b, &p.tmap_x, ks * 128, 0, full + stage);
          bulk_load(sa, p.sfw + (static_cast<size_t>(j) * (KB / 4) + 4 * ks) * 512, 512u * nkk, full + stage);
          bulk_load(sb, p.sfx + static_cast<size_t>(4 * ks) * 512, 512u * nkk, full + stage);
        }
        __syncwarp();
        filled_mask |= 1u << stage;
        fill_bits = (fill_bits & ~(1u << stage)) | (phase << stage);
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      report_timeout(p.status);
      *abort_flag = 1;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t kIdesc = idesc_mxf4nvf4(128, TN);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = 0; it < n_mine && ok && !p.test_stall; ++it) {
      const int buf = it % C::kNacc;
      const uint32_t acc_phase = (it / C::kNacc) & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(acc_empty + buf, acc_phase ^ 1u, deadline, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + buf * TN;
      for (int ks = 0; ks < k_stages; ++ks) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(full + stage, phase, deadline, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int nkk = min(4, KB / 4 - 4 * ks);
        const uint8_t* a = smem + stage * C::kStage;
        const uint8_t* sa = a + kSWTile;
        const uint8_t* b = sa + kSSfSlab;
        const uint8_t* sb = b + C::kXTile;
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
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
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
    const int et = threadIdx.x - 64;                  // 0..255
    const int quarter = warp & 3;                     // tensor-memory lanes 32 * quarter ..
    const int half = (warp - 2) >> 2;                 // token columns [half * TN / 2, (half + 1) * TN / 2)
    const int wrow = quarter * 32 + lane;             // weight row of the tile held by this thread
    const float gscale = __fmul_rn(__ldg(p.x_gsa), __ldg(p.w_gsa));
    // top-k mode: thread et takes token tok over the tile's outputs
    // [grp * OPG, grp * OPG + OPG), OPG = TN / 2 (kSEpi / TN groups)
    constexpr int OPG = TN / 2;
    constexpr int CH = OPG < 32 ? OPG : 32;           // keys per pass
    const int tok = et % TN, grp = et / TN;
    const bool tok_ok = tok < p.T;
    TopK<KMAX> tk;
    tk.init();
    unsigned long long published = 0ull;            // the list's best entry when last published
    bool ok = true;
    for (int it = 0; it < n_mine; ++it) {
      const int j = split + it * p.n_splits;
      const int buf = it % C::kNacc;
      const uint32_t acc_phase = (it / C::kNacc) & 1;
      if (!kLogits && et < 128) {
        // the previous tile's readers of s_tr / s_bias are done (barrier below)
        const int n = j * 128 + et;
        s_bias[et] = (p.bias && n < p.N) ? __ldg(p.bias + n) : 0.0f;
      }
      const bool got = bar_and(1, kSEpi, mbar_wait(acc_full + buf, acc_phase, deadline, abort_flag));
      if (!got) { ok = false; break; }
      tc_fence_after();
      const int n = j * 128 + wrow;
#pragma unroll 1
      for (int c = 0; c < OPG / CH; ++c) {
        float v[CH];
        const int t0 = half * OPG + c * CH;            // first token column of this load
        const uint32_t ta = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * TN + t0;
        if constexpr (CH == 16) tmem_load16(ta, v);
        else tmem_load32(ta, v);
        if constexpr (kLogits) {
          if (n < p.N) {
#pragma unroll
            for (int i = 0; i < CH; ++i) {
              const int t = t0 + i;
              if (t < p.T) {
                const float l = __fmul_rn(v[i], gscale);
                if (p.out_bf16)
                  reinterpret_cast<uint16_t*>(p.out)[static_cast<size_t>(t) * p.N + n] =
                      static_cast<uint16_t>(bf16_rn_bits(l));
                else
                  reinterpret_cast<float*>(p.out)[static_cast<size_t>(t) * p.N + n] = l;
              }
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < CH; ++i) s_tr[(t0 + i) * 129 + wrow] = __fmul_rn(v[i], gscale);
        }
      }
      // the accumulator may be refilled
      tc_fence_before();
      mbar_arrive(acc_empty + buf);
      if constexpr (!kLogits) {
        asm volatile("bar.sync 2, 256;" ::: "memory");      // the transposed tile is complete
        const float* row = s_tr + tok * 129 + grp * OPG;
        const int n0 = j * 128 + grp * OPG;
#pragma unroll 1
        for (int c0 = 0; c0 < OPG; c0 += CH) {
          // pass 1: keys of CH outputs and the exact k-th largest of the list
          // and the chunk together (keys-only insertion); only outputs with
          // key >= tau can enter the list
          float kv[CH];
          float sk[KMAX];
#pragma unroll
          for (int q = 0; q < KMAX; ++q) sk[q] = tk.key[q];
#pragma unroll
          for (int i = 0; i < CH; ++i) {
            const float l = row[c0 + i];
            float key = l;
            if (!p.raw) key = __fadd_rn(sigmoid_f32(l), s_bias[grp * OPG + c0 + i]);
            kv[i] = (tok_ok && n0 + c0 + i < p.N) ? key : -INFINITY;
#pragma unroll
            for (int q = KMAX - 1; q > 0; --q) sk[q] = fmaxf(sk[q], fminf(sk[q - 1], kv[i]));
            sk[0] = fmaxf(sk[0], kv[i]);
          }
          const float tau = sk[KMAX - 1];
          uint32_t cand = 0;
#pragma unroll
          for (int i = 0; i < CH; ++i) cand |= static_cast<uint32_t>(kv[i] != -INFINITY && kv[i] >= tau) << i;
          // pass 2: the candidates enter the list -- at most KMAX of them
          // plus exact ties at tau.  With an 8-entry list up to 8 are gathered
          // into fixed slots, sorted by a 19-comparator network and merged
          // with a bitonic merge (no data-dependent control flow); the rest
          // take the exact insertion in warp-uniform rounds.
          if constexpr (KMAX == 8) {
            float gk[8], gs[8];
            int gi[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              const bool has = cand != 0;
              const int i = has ? __ffs(cand) - 1 : 0;
              cand &= cand - 1;
              const float l = row[c0 + i];
              const float sc = p.raw ? l : sigmoid_f32(l);
              gk[r] = has ? (p.raw ? l : __fadd_rn(sc, s_bias[grp * OPG + c0 + i])) : -INFINITY;
              gi[r] = has ? n0 + c0 + i : 0x7FFFFFFF;
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
            const float l = row[c0 + i];
            const float sc = p.raw ? l : sigmoid_f32(l);
            const float key = p.raw ? l : __fadd_rn(sc, s_bias[grp * OPG + c0 + i]);
            tk.push_if(key, n0 + c0 + i, sc, has);
          }
        }
        asm volatile("bar.sync 2, 256;" ::: "memory");      // s_tr / s_bias are free again
        // Publish this list's best entry into the token's slots when it has
        // changed: by the time the CTAs append their candidates the slots
        // hold the best entries of every list, which bound the token's k-th
        // best tightly, and few entries per token pass.
        if (p.n_splits > 1 && tok_ok && tk.key[0] != -INFINITY) {
          const unsigned long long best = pack_key(tk.key[0], tk.id[0]);
          if (best != published) {
            atomicMax(p.tok_slots + tok * 32 + (tk.id[0] & 31), best);
            published = best;
          }
        }
      }
    }
    if (!ok) {
      report_timeout(p.status);
      *abort_flag = 1;
    }
    if constexpr (!kLogits) {
      // one abort decision for the eight epilogue warps
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (et == 0) *epi_abort = *abort_flag;
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (!*epi_abort) {
        // The token slots' words (see below) start on their way into the ring
        // now, past the lists of the group merge, so that their round trip
        // to L2 overlaps the merge: the ring is idle (every copy into it has
        // landed, since the MMAs of the last tile have read them).  The
        // snapshot is a few microseconds older than after the merge, so its
        // bound may be a little lower -- still a valid lower bound.
        unsigned long long* s_words = reinterpret_cast<unsigned long long*>(smem + 65536);
        if (p.n_splits > 1) {
          for (int i = et; i < p.T * 16; i += kSEpi)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::
                         "r"(smem_u32(reinterpret_cast<ulonglong2*>(s_words) + i)),
                         "l"(reinterpret_cast<uint64_t>(reinterpret_cast<const ulonglong2*>(p.tok_slots) + i))
                         : "memory");
          asm volatile("cp.async.commit_group;" ::: "memory");
        }
        // the kSEpi / TN groups of a token merge in a tree: in each round the
        // upper half of the groups hands its lists through shared memory (the
        // ring: every copy into it has landed, since the MMAs of the last
        // tile have read them) to the lower half, which folds them in (a
        // bitonic merge for 8-entry lists).  Entry i of every list is one
        // row, so a warp's lanes (consecutive tokens) touch consecutive
        // 16-byte words: no bank conflicts (measured at k = 8: 5.3 -> 2.5 us
        // for the three rounds).
        float4* s_l = reinterpret_cast<float4*>(smem);          // [KMAX][kSEpi / 2]
#pragma unroll 1
        for (int h = kSEpi / TN / 2; h >= 1; h >>= 1) {
          if (grp >= h && grp < 2 * h) {
#pragma unroll
            for (int i = 0; i < KMAX; ++i)
              s_l[i * (kSEpi / 2) + (grp - h) * TN + tok] =
                  make_float4(tk.key[i], __int_as_float(tk.id[i]), tk.sc[i], 0.f);
          }
          asm volatile("bar.sync 1, 256;" ::: "memory");
          if (grp < h) {
            const float4* src = s_l + grp * TN + tok;
            float bk[KMAX], bs[KMAX];
            int bi[KMAX];
#pragma unroll
            for (int i = 0; i < KMAX; ++i) {
              const float4 v = src[i * (kSEpi / 2)];
              bk[i] = v.x; bi[i] = __float_as_int(v.y); bs[i] = v.z;
            }
            tk.merge_sorted(bk, bi, bs);
          }
          asm volatile("bar.sync 1, 256;" ::: "memory");
        }
        if (p.n_splits == 1) {
          if (grp == 0 && tok_ok) {
            float sum = 0.0f;
#pragma unroll
            for (int i = 0; i < KMAX; ++i)
              if (i < p.k) sum = __fadd_rn(sum, tk.sc[i]);
#pragma unroll
            for (int i = 0; i < KMAX; ++i)
              if (i < p.k) {
                p.out_ids[tok * p.k + i] = tk.id[i];
                p.out_w[tok * p.k + i] =
                    p.raw ? tk.sc[i] : (sum > 0.0f ? __fdiv_rn(__fmul_rn(p.routed_scaling, tk.sc[i]), sum) : 0.0f);
              }
          }
        } else {
          // g, the k-th largest of the token's slot words (published by the
          // lists of every CTA as they improved), is at most the token's k-th
          // best, so an entry below g cannot be among its k best: only the
          // prefix of the sorted list at or above g is appended to the
          // token's candidates.
          // the slot words issued before the merge
          asm volatile("cp.async.wait_all;" ::: "memory");
          asm volatile("bar.sync 1, 256;" ::: "memory");
          // g of every token by rank counting, the eight warps taking tokens
          // w, w + 8, ...: lane j holds slot word j and counts the words
          // above it (the set words are distinct -- each holds a different
          // id); the set word with k - 1 above it is the k-th largest, and
          // with fewer than k set words g is 0
          unsigned long long* s_g = s_words + 128 * 32;            // [T]
          for (int t = et >> 5; t < p.T; t += kSEpi / 32) {
            const unsigned long long mine = s_words[t * 32 + lane];
            int above = 0;
#pragma unroll 8
            for (int q = 0; q < 32; ++q) above += s_words[t * 32 + q] > mine ? 1 : 0;
            const uint32_t hit = __ballot_sync(0xFFFFFFFFu, mine != 0ull && above == p.k - 1);
            const int src = hit ? __ffs(hit) - 1 : 0;
            const uint32_t lo = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(mine), src);
            const uint32_t hi = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(mine >> 32), src);
            if (lane == 0) s_g[t] = hit ? (static_cast<unsigned long long>(hi) << 32) | lo : 0ull;
          }
          asm volatile("bar.sync 1, 256;" ::: "memory");
          if (grp == 0 && tok_ok) {
            const unsigned long long g = s_g[tok];
            int n = 0;
#pragma unroll
            for (int i = 0; i < KMAX; ++i)
              if (i < p.k && tk.key[i] != -INFINITY && pack_key(tk.key[i], tk.id[i]) >= g) n = i + 1;
            const uint32_t base = atomicAdd(p.tok_count + tok, static_cast<uint32_t>(n));
            float4* dst = p.surv + static_cast<size_t>(tok) * p.surv_stride + base;
#pragma unroll
            for (int i = 0; i < KMAX; ++i)
              if (i < n) dst[i] = make_float4(tk.key[i], __int_as_float(tk.id[i]), tk.sc[i], 0.f);
          }
          // The barrier orders the epilogue threads' appends before thread
          // 0's ticket, an acquire-release atomic at gpu scope: it publishes
          // them (release, cumulative over the barrier) and, in the last
          // CTA, makes every other CTA's appends visible (acquire).
          asm volatile("bar.sync 1, 256;" ::: "memory");
          if (et == 0) {
            uint32_t old;
            asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(p.ticket) : "memory");
            *last_flag = old == static_cast<uint32_t>(p.n_splits - 1) ? 1 : 0;
          }
          asm volatile("bar.sync 1, 256;" ::: "memory");
        }
      }
    }
  }

  // --------------------------------------------- the last CTA's final merge
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (!kLogits && *last_flag) {
    __threadfence();
    // Each token's candidates (every CTA's entries at or above the bound it
    // saw: a superset of the token's k best, typically a few per k) go to
    // one warp: lane l folds candidates l, l + 32, ... into a sorted list,
    // then k rounds take the warp's best head (two 32-bit max reductions over
    // the order-preserving 64-bit (key, id) word) and the winning lane drops
    // it.
    constexpr int kWarps = kSThreads / 32;
    // every token's count and the first 32 slots of its candidates (those
    // past the count are not read later) into the (idle) ring at once: one
    // round trip to L2 for all of them
    uint32_t* s_cnt = reinterpret_cast<uint32_t*>(s_tr);                 // [T]
    float4* s_first = reinterpret_cast<float4*>(smem);                    // [T][32]
    for (int t = 4 * threadIdx.x; t < p.T; t += 4 * kSThreads)          // [128] counts: 16-byte pieces
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(s_cnt + t)),
                   "l"(reinterpret_cast<uint64_t>(p.tok_count + t)) : "memory");
    const int n_first = p.surv_stride < 32 ? p.surv_stride : 32;       // inside the token's region
    for (int i = threadIdx.x; i < p.T * 32; i += kSThreads) {
      const int t = i >> 5, j = i & 31;
      if (j < n_first)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(s_first + i)),
                     "l"(reinterpret_cast<uint64_t>(p.surv + static_cast<size_t>(t) * p.surv_stride + j))
                     : "memory");
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
    __syncthreads();
    // a warp's k winners by rank (id, score), for the sum in rank order
    float2* s_win = reinterpret_cast<float2*>(s_cnt + 128) + warp * KMAX;
#pragma unroll 1
    for (int tt = warp; tt < p.T; tt += kWarps) {
      const int cnt = static_cast<int>(s_cnt[tt]);
      if (KMAX > 1 && cnt <= 32) {
        // At most one candidate per lane (the usual case: the bound lets a
        // few per k through): each lane's rank among the token's candidates
        // (key descending, lower id first; the ids are distinct) is the
        // number of them that beat it, counted over broadcast reads -- no
        // serial rounds.  The winners land at their rank, so the weights'
        // sum runs in rank order whatever order the candidates came in.
        const float4* cand = s_first + tt * 32;
        const bool has = lane < cnt;
        const float4 v = has ? cand[lane] : make_float4(-INFINITY, 0.f, 0.f, 0.f);
        const int vid = __float_as_int(v.y);
        int rank = 0;
#pragma unroll 4
        for (int q = 0; q < cnt; ++q) {
          const float4 u = cand[q];
          rank += topk_better(u.x, __float_as_int(u.y), v.x, vid) ? 1 : 0;
        }
        if (has && rank < p.k) s_win[rank] = make_float2(__int_as_float(vid), v.z);
        __syncwarp();
        const bool mine = lane < p.k && lane < cnt;
        const float2 w = mine ? s_win[lane] : make_float2(__int_as_float(0x7FFFFFFF), 0.f);
        float sum = mine ? w.y : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xFFFFFFFFu, sum, o));
        if (lane < p.k) {
          p.out_ids[tt * p.k + lane] = __float_as_int(w.x);
          p.out_w[tt * p.k + lane] =
              p.raw ? w.y : (sum > 0.0f ? __fdiv_rn(__fmul_rn(p.routed_scaling, w.y), sum) : 0.0f);
        }
        if (lane == 0) p.tok_count[tt] = 0u;
        __syncwarp();                                  // s_win is reused by the warp's next token
        continue;
      }
      TopK<KMAX> mine;
      mine.init();
      if (lane < cnt) {
        const float4 v = s_first[tt * 32 + lane];
        mine.push(v.x, __float_as_int(v.y), v.z);
      }
      for (int j = lane + 32; j < cnt; j += 32) {
        const float4 v = __ldcg(p.surv + static_cast<size_t>(tt) * p.surv_stride + j);
        mine.push(v.x, __float_as_int(v.y), v.z);
      }
      float key = -INFINITY, sc = 0.0f;
      int id = 0x7FFFFFFF;
#pragma unroll 1
      for (int r = 0; r < p.k; ++r) {
        const uint64_t w = mine.key[0] == -INFINITY ? 0ull : pack_key(mine.key[0], mine.id[0]);
        const uint32_t hi = static_cast<uint32_t>(w >> 32), lo = static_cast<uint32_t>(w);
        const uint32_t hmax = __reduce_max_sync(0xFFFFFFFFu, hi);
        const uint32_t lmax = __reduce_max_sync(0xFFFFFFFFu, hi == hmax ? lo : 0u);
        const bool win = w != 0ull && hi == hmax && lo == lmax;
        const int src = __ffs(__ballot_sync(0xFFFFFFFFu, win)) - 1;
        const float wk = __shfl_sync(0xFFFFFFFFu, mine.key[0], src < 0 ? 0 : src);
        const int wi = __shfl_sync(0xFFFFFFFFu, mine.id[0], src < 0 ? 0 : src);
        const float ws = __shfl_sync(0xFFFFFFFFu, mine.sc[0], src < 0 ? 0 : src);
        if (lane == r && src >= 0) { key = wk; id = wi; sc = ws; }
        if (win) mine.pop_front();
      }
      float sum = lane < p.k ? sc : 0.0f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xFFFFFFFFu, sum, o));
      if (lane < p.k) {
        p.out_ids[tt * p.k + lane] = id;
        p.out_w[tt * p.k + lane] =
            p.raw ? sc : (sum > 0.0f ? __fdiv_rn(__fmul_rn(p.routed_scaling, sc), sum) : 0.0f);
      }
      if (lane == 0) p.tok_count[tt] = 0u;
    }
    for (int i = threadIdx.x; i < p.T * 32; i += kSThreads) p.tok_slots[i] = 0ull;
    if (threadIdx.x == 0) *p.ticket = 0u;
  }

  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // copies may still be landing in shared memory: wait (bounded) for the
    // latest fill of every ring stage before the CTA exits
    const uint64_t drain = globaltimer_ns() + 1000000000ull;
    for (int s = 0; s < C::kStages; ++s) {
      if (!((filled_mask >> s) & 1u)) continue;
      while (!mbar_try_wait(full + s, (fill_bits >> s) & 1u))
        if (globaltimer_ns() > drain) break;
    }
  }
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int TN, int KMAX, bool kLogits>
cudaError_t launch_stream_k(const StreamParams& p, int grid, cudaStream_t s) {
  using C = StreamCfg<TN>;
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(gemm_stream_kernel<TN, KMAX, kLogits>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_stream_kernel<TN, KMAX, kLogits>, p);
}

template <int TN>
cudaError_t launch_stream_tn(const StreamParams& p, int grid, bool logits, int k, cudaStream_t s) {
  if (logits) return launch_stream_k<TN, 1, true>(p, grid, s);
  if (k <= 1) return launch_stream_k<TN, 1, false>(p, grid, s);
  if (k <= 2) return launch_stream_k<TN, 2, false>(p, grid, s);
  if (k <= 4) return launch_stream_k<TN, 4, false>(p, grid, s);
  if (k <= 8) return launch_stream_k<TN, 8, false>(p, grid, s);
  return launch_stream_k<TN, 16, false>(p, grid, s);
}

bool encode_rows_map(CUtensorMap* map, const uint8_t* ptr, int64_t rows, int64_t D, uint32_t box_rows) {
  return encode_codes(map, ptr, rows, D, box_rows);
}

}  // namespace

int stream_token_tile(int64_t T) { return T <= 32 ? 32 : (T <= 64 ? 64 : 128); }

int stream_splits(int64_t N, int num_sms) {
  const int64_t tiles = (N + 127) / 128;
  int s = num_sms > 0 ? num_sms : 1;
  if (s > tiles) s = static_cast<int>(tiles);
  if (s > kMaxSplits) s = kMaxSplits;
  return s < 1 ? 1 : s;
}

nvr_status launch_gemm_stream(const uint8_t* x_codes, const uint8_t* x_sf, const float* x_gsa, int64_t T, int64_t D,
                              const uint8_t* W_codes, const uint8_t* W_sf, const float* w_gsa, int64_t N,
                              const float* bias, int k, float routed_scaling, bool raw, int32_t* out_ids,
                              float* out_w, void* out, bool out_bf16, float4* partials, uint32_t* ticket,
                              uint32_t* status, int n_splits, bool test_stall, cudaStream_t s) {
  if (T < 1 || T > 128) return NVR_ERR_UNSUPPORTED;
  const int TN = stream_token_tile(T);
  const bool logits = out != nullptr;
  StreamParams p;
  if (!encode_rows_map(&p.tmap_w, W_codes, N, D, 128)) return NVR_ERR_UNSUPPORTED;
  if (!encode_rows_map(&p.tmap_x, x_codes, T, D, static_cast<uint32_t>(TN))) return NVR_ERR_UNSUPPORTED;
  p.sfw = W_sf; p.sfx = x_sf; p.x_gsa = x_gsa; p.w_gsa = w_gsa; p.bias = raw ? nullptr : bias;
  p.T = static_cast<int>(T); p.N = static_cast<int>(N); p.D = static_cast<int>(D); p.k = k;
  p.raw = raw ? 1 : 0; p.n_splits = n_splits; p.n_tiles = static_cast<int>((N + 127) / 128);
  p.routed_scaling = routed_scaling;
  p.out_ids = out_ids; p.out_w = out_w; p.out = out; p.out_bf16 = out_bf16 ? 1 : 0;
  p.surv = partials; p.surv_stride = n_splits * k;
  p.ticket = ticket; p.tok_count = ticket + 64; p.tok_slots = reinterpret_cast<unsigned long long*>(ticket + 512);
  p.status = status;
  p.test_stall = test_stall ? 1 : 0;
  cudaError_t e;
  if (TN == 32) e = launch_stream_tn<32>(p, n_splits, logits, k, s);
  else if (TN == 64) e = launch_stream_tn<64>(p, n_splits, logits, k, s);
  else e = launch_stream_tn<128>(p, n_splits, logits, k, s);
  return cuda_status(e);
}

}  // namespace nvr
