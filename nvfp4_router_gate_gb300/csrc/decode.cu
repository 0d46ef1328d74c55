// decode.cu -- the whole router call for a few tokens in ONE kernel launch.
//
// Source: the fused decode kernel notes of "nvfp4-megamoe-kernel commit e0f60b9:
// dsv4/kernels/router/__init__.py" (decode latency, the logits' round trip
// through memory, the row-level top-k) and the launch count of "commit 04cf8ca:
// dsv4/layers/router.py" (GEMM + activation_topk as 2 launches instead of 1).
//
// For T <= 16 tokens the gate GEMM is a skinny GEMV that streams the 1 MB
// weight once; tensor cores buy nothing at this size, latency is everything.
// Every CTA:
//   1. reduces max|x| over the whole (small) x -- the same exact maximum the
//      grid-wide amax kernel finds, so gsa has identical bits;
//   2. quantizes all of x into shared memory with the block quantizer shared
//      with the quantize kernel (identical codes and scales), keeping each
//      block as 16 signed bytes 2*e2m1(code) and its fp32 scale;
//   (for several tokens the CTAs form clusters of 4 that split steps 1-2:
//   each stages, reduces and quantizes a quarter of x and stores its blocks
//   into the other CTAs' shared memory; one token: every CTA does all of it)
//   3. computes the logits of its `epc` experts: integer dot products of each
//      16-element block (dp4a on 2*e2m1 values, exact) scaled by the two block
//      scales (exact product) and accumulated in fp32, then x gsa_x * gsa_w;
//   4. writes sigmoid scores and biased keys of its experts to the workspace.
// The last CTA to finish (atomic ticket; nobody waits) ranks each token's N
// keys (key descending, lower id first), renormalises the k selected scores
// and writes ids and weights, then resets the ticket.
#include "nvr_internal.h"
#include "nvr_tcgen05.cuh"

namespace nvr {

constexpr int kDecodeThreads = 512;
// Several tokens: clusters of 4 CTAs share the staging and quantization of x.
// (Measured on GB300: clusters of 8 were launched in waves, several µs apart;
// for a single token the cluster barriers cost more than the sharing saves.)
constexpr int kMaxDecodeCluster = 4;
constexpr int kDecodeWarps = kDecodeThreads / 32;

struct DecodeParams {
  const void* x;
  int T, D;
  const uint8_t* W_codes;
  const uint8_t* W_sf;
  const float* w_gsa;
  int N;
  const float* bias;
  int k;
  float routed_scaling;
  int raw, epc;
  int32_t* out_ids;
  float* out_w;
  float* logits;
  float* ws_keys;
  float* ws_scores;
  uint32_t* ticket;
  // null: the last CTA (ticket) collects the keys; else (N <= 256) the
  // collector words of every (token, expert) pair, zero between calls
  uint64_t* ws_words;
  uint32_t* status;            // timeout of the collector's poll, or null
  int test_stall;              // test hook: CTAs other than the collector store no words
  // CTAs per thread-block cluster (1: every CTA stages, reduces and
  // quantizes all of x itself; C > 1: the C CTAs of a cluster split these
  // and exchange the results through distributed shared memory)
  int cluster;
};

// Four E2M1 codes (16 bits, element i in nibble i) -> four signed bytes
// holding 2 * value (0, +-1, +-2, +-3, +-4, +-6, +-8, +-12).
__device__ __forceinline__ uint32_t e2m1x4_to_s8x4(uint32_t c16) {
  uint32_t mag;
  // byte permute as an 8-entry table: magnitudes of codes 0..7 times two
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(mag) : "r"(0x03020100u), "r"(0x0C080604u), "r"(c16 & 0x7777u));
  const uint32_t neg = (0x80808080u - mag) ^ 0x80808080u;     // per-byte negation, no carries
  const uint32_t sb = ((c16 & 0x0008u) << 4) | ((c16 & 0x0080u) << 8) | ((c16 & 0x0800u) << 12) |
                      ((c16 & 0x8000u) << 16);
  const uint32_t mask = (sb >> 7) * 0xFFu;
  return (mag & ~mask) | (neg & mask);
}

// (key descending, id ascending) as one unsigned 64-bit order: the float's
// order-preserving bit pattern above the complemented id; 0 marks "none".
__device__ __forceinline__ uint64_t dec_pack_key(float key, int id) {
  const uint32_t b = __float_as_uint(key);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(id));
}

constexpr int kCandCap = 64;

// A collector word: the key's order-preserving bits (never 0: a word of 0
// means "not written yet") above the score's bits.
__device__ __forceinline__ uint64_t dec_word(float key, float score) {
  const uint32_t b = __float_as_uint(key);
  uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  ord = ord > 1u ? ord : 1u;                       // only a NaN pattern maps to 0
  return (static_cast<uint64_t>(ord) << 32) | __float_as_uint(score);
}
__device__ __forceinline__ float dec_word_key(uint64_t w) {
  const uint32_t ord = static_cast<uint32_t>(w >> 32);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Top-k (k <= 16) of one token's N <= 256 keys with one warp, in order (key
// descending, lower id first): lane l holds keys l, l+32, ...  The k-th
// largest of the 32 lane maxima is a lower bound of the k-th largest key (the
// k largest maxima are k keys at least that large), so only keys >= it are
// candidates -- typically k to 2k -- and each candidate's rank among the
// candidates is its rank overall.
// More than kCandCap candidates (exact ties) fall back to k rounds of a warp
// arg-max.  sel[r] receives the expert of rank r; cand is warp scratch.
__device__ __forceinline__ void warp_topk_256(const float* kt, int N, int k, int lane, uint64_t* cand, int* sel) {
  uint64_t pk[8];
  uint64_t mx = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int n = lane + 32 * j;
    pk[j] = n < N ? dec_pack_key(kt[n], n) : 0;
    mx = pk[j] > mx ? pk[j] : mx;
  }
  // the k-th largest lane maximum: the k largest maxima are k keys at least
  // that large (0 when fewer than k lanes hold keys: every key is a candidate)
  cand[lane] = mx;
  __syncwarp();
  int mrank = 0;
#pragma unroll 8
  for (int q = 0; q < 32; ++q) mrank += cand[q] > mx ? 1 : 0;
  const uint32_t at_k = __ballot_sync(0xFFFFFFFFu, mx != 0 && mrank == k - 1);
  const uint64_t bound = at_k ? __shfl_sync(0xFFFFFFFFu, mx, __ffs(at_k) - 1) : 0;
  __syncwarp();                                    // cand is rewritten below
  uint32_t cmask = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) cmask |= static_cast<uint32_t>(pk[j] != 0 && pk[j] >= bound) << j;
  const int cnt = __popc(cmask);
  int incl = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += y;
  }
  const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  if (total <= kCandCap) {
    int pos = incl - cnt;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if ((cmask >> j) & 1u) cand[pos++] = pk[j];
    __syncwarp();
    for (int ci = lane; ci < total; ci += 32) {
      const uint64_t me = cand[ci];
      int rk = 0;
      for (int q = 0; q < total; ++q) rk += cand[q] > me ? 1 : 0;
      if (rk < k) sel[rk] = static_cast<int>(~static_cast<uint32_t>(me));
    }
  } else {
    // many equal keys: k rounds of a warp arg-max, the winner's key removed
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
      uint64_t m = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) m = pk[j] > m ? pk[j] : m;
      const uint32_t hmax = __reduce_max_sync(0xFFFFFFFFu, static_cast<uint32_t>(m >> 32));
      const uint32_t lmax = __reduce_max_sync(0xFFFFFFFFu, static_cast<uint32_t>(m >> 32) == hmax
                                                               ? static_cast<uint32_t>(m) : 0u);
      const uint64_t w = (static_cast<uint64_t>(hmax) << 32) | lmax;
#pragma unroll
      for (int j = 0; j < 8; ++j) pk[j] = pk[j] == w ? 0 : pk[j];
      if (lane == 0) sel[r] = static_cast<int>(~lmax);
    }
  }
  __syncwarp();
}

__host__ __device__ constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr int kMaxBlocksPerThread = 8;    // W blocks a thread prefetches into registers
constexpr size_t kCollectBytes = 4096;    // shared memory of the one-token collector
constexpr int kMaxT = 16;                 // tokens of one decode call

// Shared memory of one CTA: the raw activations (reused for the last CTA's
// keys and scores), their signed 2*e2m1 bytes, their block scales and the
// cross-warp partial sums.
struct DecodeSmem {
  size_t raw, xv, xs, red, total;
};
__host__ __device__ inline DecodeSmem decode_smem_layout(int T, int D, int N, int elt, int C) {
  const int KB = D / kBlock;
  DecodeSmem L;
  L.raw = 0;
  // the raw activations of this CTA's blocks only: all of x, or a cluster
  // rank's slice
  const size_t slice = (static_cast<size_t>(T) * KB + C - 1) / C;
  const size_t raw_bytes = slice * kBlock * elt;
  const size_t kv_bytes = static_cast<size_t>(T) * N * 8;
  // (at least the one-token collector's 4 KB: 256 order words, 256 scores
  // and 128 candidates, clear of the regions still read before it starts)
  size_t xr = raw_bytes > kv_bytes ? raw_bytes : kv_bytes;
  xr = xr > kCollectBytes ? xr : kCollectBytes;
  L.xv = align_up(xr, 16);
  L.xs = align_up(L.xv + static_cast<size_t>(T) * D, 16);
  L.red = align_up(L.xs + static_cast<size_t>(T) * KB * 4, 16);
  // cross-warp partial sums, later the last CTA's candidate lists (8 B each)
  const size_t red_bytes = static_cast<size_t>(kDecodeWarps) * kMaxT * 4;
  const size_t cand_bytes = static_cast<size_t>(kDecodeWarps) * kCandCap * 8;
  L.total = L.red + (red_bytes > cand_bytes ? red_bytes : cand_bytes);
  return L;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(smem_dst)),
               "l"(reinterpret_cast<uint64_t>(gmem_src)) : "memory");
}

// Distributed shared memory: the address of a local shared-memory location in
// CTA `rank` of the cluster, and stores to it.
__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, const uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}

template <bool kBF16>
__global__ void __launch_bounds__(kDecodeThreads, 1)
decode_router_kernel(const DecodeParams p) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int T = p.T, D = p.D, N = p.N, KB = D / kBlock;
  const DecodeSmem L = decode_smem_layout(T, D, N, kBF16 ? 2 : 4, p.cluster);
  uint8_t* xraw = sm + L.raw;
  int8_t* xv = reinterpret_cast<int8_t*>(sm + L.xv);
  float* xs = reinterpret_cast<float*>(sm + L.xs);
  float* red = reinterpret_cast<float*>(sm + L.red);          // [warps][kMaxT]
  __shared__ uint32_t s_red[kDecodeWarps];
  __shared__ uint32_t s_cmax[kMaxDecodeCluster];
  __shared__ int s_last;
  __shared__ int s_sel[kMaxT * 16];
  __shared__ float s_rcp[128];                                   // RN(1 / dec(b)) of scale byte b

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gs = kDecodeThreads / p.epc;                       // threads per expert
  const int grp = tid / gs, j = tid - grp * gs;
  const int e = blockIdx.x * p.epc + grp;

  // slots i with i * gs < KB hold blocks (the bound is the same in every
  // thread, so the unrolled loops below skip the empty slots with a uniform
  // branch instead of computing on them)
  const int nb = (KB + gs - 1) / gs;
  // The launch may overlap the previous kernel of the stream (programmatic
  // dependent launch), which may still be writing x, W or the workspace.
  // Until it has finished only L2 prefetches of this thread's weight blocks
  // are issued: they return nothing to the thread, and L2 is where every
  // write lands, so a prefetched line is never stale.
#pragma unroll
  for (int i = 0; i < kMaxBlocksPerThread; ++i) {
    const int c = j + i * gs;
    if (i >= nb) break;
    if (e < N && c < KB) {
      asm volatile("prefetch.global.L2 [%0];" :: "l"(p.W_codes + static_cast<size_t>(e) * (D / 2) + c * 8));
      asm volatile("prefetch.global.L2 [%0];" :: "l"(p.W_sf + sf_tile_offset(e, c, KB)));
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next kernel of the stream may launch now; it waits for this grid to
  // complete before it reads anything
  asm volatile("griddepcontrol.launch_dependents;");

  // 0. Load this thread's weight blocks into registers (independent of x;
  //    their latency overlaps everything up to the dot products) and stage x
  //    in shared memory with one burst of asynchronous 16-byte copies.
  uint2 wc[kMaxBlocksPerThread];
  uint32_t wsb[kMaxBlocksPerThread];
#pragma unroll
  for (int i = 0; i < kMaxBlocksPerThread; ++i) {
    const int c = j + i * gs;
    if (i >= nb) break;
    if (e < N && c < KB) {
      wc[i] = __ldg(reinterpret_cast<const uint2*>(p.W_codes + static_cast<size_t>(e) * (D / 2) + c * 8));
      wsb[i] = __ldg(p.W_sf + sf_tile_offset(e, c, KB));
    } else {
      wc[i] = make_uint2(0, 0);
      wsb[i] = 0;
    }
  }
  // The threads that finish an expert's logit (step 4) load the gate's global
  // scale and the expert's bias now, off the path to the keys.
  const int g_out = tid / kMaxT, t_out = tid - g_out * kMaxT;
  const int e_out = blockIdx.x * p.epc + g_out;
  const bool out_thread = tid < p.epc * kMaxT && t_out < T && e_out < N;
  float w_gsa = 0.0f, bias_e = 0.0f;
  if (out_thread) {
    w_gsa = __ldg(p.w_gsa);
    if (p.bias) bias_e = __ldg(p.bias + e_out);
  }
  // The blocks of x (block b = t * KB + c: 16 elements of token t) this CTA
  // stages, reduces and quantizes: all of them, or in a cluster of C CTAs
  // the slice [b_lo, b_hi) of its rank.
  const int C = p.cluster;
  uint32_t crank = 0;
  if (C > 1) {
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
    // distributed shared memory may be accessed once every CTA of the
    // cluster runs: arrive now, wait before the first remote store
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  }
  const int nblk = T * KB;
  int b_lo = 0, b_hi = nblk;
  if (C > 1) {
    const int per = (nblk + C - 1) / C;
    b_lo = min(nblk, static_cast<int>(crank) * per);
    b_hi = min(nblk, b_lo + per);
  }
  constexpr int kVecPerBlock = kBlock * (kBF16 ? 2 : 4) / 16;     // 16-byte vectors per block
  for (int v = b_lo * kVecPerBlock + tid; v < b_hi * kVecPerBlock; v += kDecodeThreads)
    cp_async16(xraw + 16 * static_cast<size_t>(v - b_lo * kVecPerBlock),
               static_cast<const uint8_t*>(p.x) + 16 * static_cast<size_t>(v));
  asm volatile("cp.async.commit_group;" ::: "memory");
  // the quantizer's reciprocal table (the bits __frcp_rn gives), while the
  // copies are in flight; byte 127 (NaN) never occurs
  if (tid < 128) s_rcp[tid] = (tid >= 1 && tid <= 126) ? __frcp_rn(e4m3_value(tid)) : 0.0f;
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  // 1. max |x| over the staged blocks; in a cluster, every CTA's maximum goes
  //    to every CTA (thread i writes CTA i's slot), so each one finds the
  //    maximum of the whole batch -- the same exact value in every CTA
  const uint4* x4 = reinterpret_cast<const uint4*>(xraw);
  uint32_t m = 0;
  for (int v = tid; v < (b_hi - b_lo) * kVecPerBlock; v += kDecodeThreads) m = max(m, absmax_bits16B<kBF16>(x4[v]));
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if (lane == 0) s_red[warp] = m;
  __syncthreads();
  static_assert(kDecodeWarps <= 32, "one warp reduces the warps' maxima");
  uint32_t mb = __reduce_max_sync(0xFFFFFFFFu, lane < kDecodeWarps ? s_red[lane] : 0u);
  if (C > 1) {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (tid < C) st_cluster_u32(cluster_addr(s_cmax + crank, tid), mb);
    cluster_sync_all();
    mb = 0;
    for (int r = 0; r < C; ++r) mb = max(mb, s_cmax[r]);
  }
  const QuantScale qs = make_quant_scale(__uint_as_float(mb));

  // 2. quantize the blocks (shared -> shared) with the block quantizer shared
  //    with the quantize kernel: identical codes and scales.  Block b keeps
  //    its 16 signed bytes at xv + 16 b and its scale at xs[b]; in a cluster
  //    each CTA also stores its blocks into every other CTA's copy.
  for (int b = b_lo + tid; b < b_hi; b += kDecodeThreads) {
    Block16 blk;
    load_block16_shared<kBF16>(xraw, static_cast<size_t>(b - b_lo) * kBlock, blk);   // xraw holds [b_lo, b_hi)
    uint32_t lo, hi;
    const uint32_t byte = quant_block16_bracket(blk, qs, lo, hi, s_rcp);
    uint4 q;
    q.x = e2m1x4_to_s8x4(lo & 0xFFFFu);
    q.y = e2m1x4_to_s8x4(lo >> 16);
    q.z = e2m1x4_to_s8x4(hi & 0xFFFFu);
    q.w = e2m1x4_to_s8x4(hi >> 16);
    const float sc = e4m3_value(byte);
    *reinterpret_cast<uint4*>(xv + 16 * static_cast<size_t>(b)) = q;
    xs[b] = sc;
    for (int r = 1; r < C; ++r) {
      const uint32_t peer = (crank + r) % C;                     // a different peer per step
      st_cluster_v4(cluster_addr(xv + 16 * static_cast<size_t>(b), peer), q);
      st_cluster_u32(cluster_addr(xs + b, peer), __float_as_uint(sc));
    }
  }
  // every block in every CTA of the cluster (and no remote access after)
  if (C > 1) cluster_sync_all();
  else __syncthreads();

  // decode this thread's weight blocks: their loads were issued first and have
  // long landed; decoding them only now keeps them off the path to gsa
  uint32_t wv[kMaxBlocksPerThread][4];
  float swv[kMaxBlocksPerThread];
#pragma unroll
  for (int i = 0; i < kMaxBlocksPerThread; ++i) {
    if (i >= nb) break;
    swv[i] = e4m3_value(wsb[i]);
    wv[i][0] = e2m1x4_to_s8x4(wc[i].x & 0xFFFFu);
    wv[i][1] = e2m1x4_to_s8x4(wc[i].x >> 16);
    wv[i][2] = e2m1x4_to_s8x4(wc[i].y & 0xFFFFu);
    wv[i][3] = e2m1x4_to_s8x4(wc[i].y >> 16);
  }

  // 3. logits of this CTA's experts: integer dot products of each 16-element
  //    block (exact), scaled by the two block scales (exact product), fp32 sum.
  //    The weight blocks are decoded once; the token loop stays rolled.
  // Four tokens at a time (one for a single token): their block loops and
  // warp reductions interleave; a token's own sums keep the block order, so
  // results do not depend on T.
  if (T == 1) {
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxBlocksPerThread; ++i) {
      const int c = j + i * gs;
      if (i >= nb) break;
      if (e < N && c < KB) {
        const uint4 xq = *reinterpret_cast<const uint4*>(xv + c * kBlock);
        int sdot = __dp4a(static_cast<int>(xq.x), static_cast<int>(wv[i][0]), 0);
        sdot = __dp4a(static_cast<int>(xq.y), static_cast<int>(wv[i][1]), sdot);
        sdot = __dp4a(static_cast<int>(xq.z), static_cast<int>(wv[i][2]), sdot);
        sdot = __dp4a(static_cast<int>(xq.w), static_cast<int>(wv[i][3]), sdot);
        acc = __fmaf_rn(static_cast<float>(sdot), __fmul_rn(xs[c], swv[i]), acc);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) red[warp * kMaxT] = acc;
  }
#pragma unroll 1
  for (int t0 = 0; t0 < (T > 1 ? T : 0); t0 += 4) {
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < kMaxBlocksPerThread; ++i) {
      const int c = j + i * gs;
      if (i >= nb) break;
      if (e < N && c < KB) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = min(t0 + u, T - 1);               // a repeated token past T is discarded
          const uint4 xq = *reinterpret_cast<const uint4*>(xv + static_cast<size_t>(t) * D + c * kBlock);
          int sdot = __dp4a(static_cast<int>(xq.x), static_cast<int>(wv[i][0]), 0);
          sdot = __dp4a(static_cast<int>(xq.y), static_cast<int>(wv[i][1]), sdot);
          sdot = __dp4a(static_cast<int>(xq.z), static_cast<int>(wv[i][2]), sdot);
          sdot = __dp4a(static_cast<int>(xq.w), static_cast<int>(wv[i][3]), sdot);
          // |sdot| <= 16 * 144 and both scales have 4 significant bits: the
          // product is exact, only the accumulation rounds
          acc[u] = __fmaf_rn(static_cast<float>(sdot), __fmul_rn(xs[t * KB + c], swv[i]), acc[u]);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[u] += __shfl_xor_sync(0xFFFFFFFFu, acc[u], o);
    if (lane == 0)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (t0 + u < T) red[warp * kMaxT + t0 + u] = acc[u];
  }
  __syncthreads();

  // 4. per (expert, token): logit, score, key
  if (out_thread) {
    const int g = g_out, t = t_out, e2 = e_out;
    const int wpg = kDecodeWarps / p.epc;
    float sacc = 0.0f;
    for (int w = 0; w < wpg; ++w) sacc = __fadd_rn(sacc, red[(g * wpg + w) * kMaxT + t]);
    const float gscale = __fmul_rn(qs.gsa, w_gsa);
    const float l = __fmul_rn(__fmul_rn(sacc, 0.25f), gscale);     // the sums count 2a * 2b
    const size_t o = static_cast<size_t>(t) * N + e2;
    if (p.logits) {
      p.logits[o] = l;
    } else {
      const float sc = p.raw ? l : sigmoid_f32(l);
      const float key = p.bias ? __fadd_rn(sc, bias_e) : sc;
      if (p.ws_words) {
        if (!p.test_stall || blockIdx.x == 0) st_relaxed_u64(p.ws_words + o, dec_word(key, sc));
      } else {
        p.ws_keys[o] = key;
        p.ws_scores[o] = sc;
      }
    }
  }
  if (p.logits) return;

  // 5. one CTA selects, renormalises and writes
  float* kbuf = reinterpret_cast<float*>(xraw);                 // x is no longer needed
  float* sbuf = kbuf + static_cast<size_t>(T) * N;
  if (p.ws_words) {
    // Up to 256 experts: CTA 0 collects.  Every other CTA has stored its
    // words and exits without waiting; CTA 0 polls the T x N words (each
    // thread up to eight, all its loads in flight at once) until none is
    // zero -- the data is its own flag, so the last word is seen about one
    // round trip after it lands, with no ticket and no second read -- and
    // puts each back to zero for the next call (nothing else writes it in
    // this call).  The poll is bounded (1 s; a timeout goes to the status
    // word and leaves the outputs unspecified).
    if (blockIdx.x != 0) return;
    constexpr int kPoll = kDecodeWords / kDecodeThreads;
    const int nw = T * N;
    uint64_t wv[kPoll];
#pragma unroll
    for (int u = 0; u < kPoll; ++u) {
      const int i = tid + u * kDecodeThreads;
      wv[u] = i < nw ? ld_relaxed_u64(p.ws_words + i) : 1ull;
    }
    const uint64_t deadline = globaltimer_ns() + 1000000000ull;
    for (;;) {
      bool all = true;
#pragma unroll
      for (int u = 0; u < kPoll; ++u) all = all && wv[u] != 0;
      if (all) break;
      if (globaltimer_ns() > deadline) {
        report_timeout(p.status);
        break;
      }
#pragma unroll
      for (int u = 0; u < kPoll; ++u)
        if (wv[u] == 0) wv[u] = ld_relaxed_u64(p.ws_words + tid + u * kDecodeThreads);
    }
#pragma unroll
    for (int u = 0; u < kPoll; ++u) {
      const int i = tid + u * kDecodeThreads;
      if (i < nw) st_relaxed_u64(p.ws_words + i, 0ull);
    }
    if (T == 1) {
      // One token: eight warps rank 32 keys each among themselves (the k best
      // of every warp are candidates: the k best overall are among them), then
      // each of the 8k candidates is ranked among the candidates; ranks follow
      // (key descending, lower id first).
      uint64_t* s_pk = reinterpret_cast<uint64_t*>(xraw);                 // [256] order words
      float* s_sc = reinterpret_cast<float*>(xraw + 256 * 8);              // [256] scores
      uint64_t* s_cand = reinterpret_cast<uint64_t*>(xraw + 256 * 12);     // [8 k]
      const int k = p.k;
      if (warp < 8) {
        const uint64_t r = tid < N ? ((wv[0] >> 32) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(tid)) : 0ull;
        if (tid < N) s_sc[tid] = __uint_as_float(static_cast<uint32_t>(wv[0]));
        s_pk[tid] = r;
        if (lane < k) s_cand[warp * k + lane] = 0ull;
        __syncwarp();
        int rk = 0;
#pragma unroll
        for (int q = 0; q < 32; ++q) rk += s_pk[warp * 32 + q] > r ? 1 : 0;
        if (r != 0 && rk < k) s_cand[warp * k + rk] = r;
      }
      __syncthreads();
      // each candidate is ranked by eight threads at once (consecutive lanes),
      // each counting the better ones among an eighth of the candidates
      // (measured at T = 1: 0.40 us, against 0.67 us with one thread per
      // candidate)
      const int nc = 8 * k;
      for (int c0 = 0; c0 < nc; c0 += kDecodeThreads / 8) {
        const int ci = c0 + (tid >> 3), part = tid & 7;
        const uint64_t c = ci < nc ? s_cand[ci] : 0ull;
        int rk = 0;
        if (ci < nc)
          for (int q = part; q < nc; q += 8) rk += s_cand[q] > c ? 1 : 0;
        rk += __shfl_xor_sync(0xFFFFFFFFu, rk, 1);
        rk += __shfl_xor_sync(0xFFFFFFFFu, rk, 2);
        rk += __shfl_xor_sync(0xFFFFFFFFu, rk, 4);
        if (part == 0 && c != 0 && rk < k) s_sel[rk] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(c));
      }
      __syncthreads();
      if (warp == 0) {
        const int id = lane < k ? s_sel[lane] : 0;
        const float sc = lane < k ? s_sc[id & 255] : 0.0f;
        float sum = sc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xFFFFFFFFu, sum, o));
        if (lane < k) {
          p.out_ids[lane] = id;
          p.out_w[lane] = p.raw ? sc : (sum > 0.0f ? __fdiv_rn(__fmul_rn(p.routed_scaling, sc), sum) : 0.0f);
        }
      }
      return;
    }
#pragma unroll
    for (int u = 0; u < kPoll; ++u) {
      const int i = tid + u * kDecodeThreads;
      if (i < nw) {
        kbuf[i] = dec_word_key(wv[u]);
        sbuf[i] = __uint_as_float(static_cast<uint32_t>(wv[u]));
      }
    }
    __syncthreads();
  } else {
    // The last CTA to finish collects.  The CTA barrier orders every
    // thread's key stores before thread 0's ticket, an acquire-release atomic
    // at gpu scope: it publishes them (release, cumulative over the barrier)
    // and, in the last CTA, makes every other CTA's published keys visible to
    // the threads that read them after the next barrier (acquire) -- one
    // round trip instead of a fence and an atomic.
    __syncthreads();
    if (tid == 0) {
      uint32_t old;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(p.ticket) : "memory");
      s_last = old == gridDim.x - 1 ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    for (int i = tid; i < T * N; i += kDecodeThreads) {
      kbuf[i] = __ldcg(p.ws_keys + i);
      sbuf[i] = __ldcg(p.ws_scores + i);
    }
    __syncthreads();
  }
  if (N <= 256) {
    // one warp per token: candidate selection, then the renormalised weights
    uint64_t* cand = reinterpret_cast<uint64_t*>(red) + warp * kCandCap;   // red is no longer needed
    for (int t = warp; t < T; t += kDecodeWarps) {
      int* sel = s_sel + t * 16;
      warp_topk_256(kbuf + static_cast<size_t>(t) * N, N, p.k, lane, cand, sel);
      const float* st = sbuf + static_cast<size_t>(t) * N;
      const float sc = lane < p.k ? st[sel[lane] & 255] : 0.0f;
      float sum = sc;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xFFFFFFFFu, sum, o));
      if (lane < p.k) {
        p.out_ids[static_cast<size_t>(t) * p.k + lane] = sel[lane];
        p.out_w[static_cast<size_t>(t) * p.k + lane] =
            p.raw ? sc : (sum > 0.0f ? __fdiv_rn(__fmul_rn(p.routed_scaling, sc), sum) : 0.0f);
      }
    }
    if (tid == 0 && !p.ws_words) *p.ticket = 0u;
    return;
  }
  if (T * N <= kDecodeThreads) {
    // Small batches: every thread ranks at most one (token, expert) key
    // against the token's N keys (key descending, lower id first); the k
    // lowest ranks are the selection, in order.
    for (int pr = tid; pr < T * N; pr += kDecodeThreads) {
      const int t = pr / N, n = pr - t * N;
      const float* kt = kbuf + static_cast<size_t>(t) * N;
      const float kn = kt[n];
      int rank = 0;
      int q = 0;
      for (; q + 8 <= N; q += 8) {                 // 8 independent shared loads per step
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float kq = kt[q + u];
          rank += (kq > kn || (kq == kn && q + u < n)) ? 1 : 0;
        }
      }
      for (; q < N; ++q) {
        const float kq = kt[q];
        rank += (kq > kn || (kq == kn && q < n)) ? 1 : 0;
      }
      if (rank < p.k) s_sel[t * 16 + rank] = n;
    }
    __syncthreads();
    if (tid < T) {
      const int t = tid;
      const float* st = sbuf + static_cast<size_t>(t) * N;
      float sum = 0.0f;
      for (int r = 0; r < p.k; ++r) sum = __fadd_rn(sum, st[s_sel[t * 16 + r]]);
      for (int r = 0; r < p.k; ++r) {
        const int n = s_sel[t * 16 + r];
        const float sc = st[n];
        p.out_ids[static_cast<size_t>(t) * p.k + r] = n;
        p.out_w[static_cast<size_t>(t) * p.k + r] =
            p.raw ? sc : (sum > 0.0f ? __fdiv_rn(__fmul_rn(p.routed_scaling, sc), sum) : 0.0f);
      }
    }
    if (tid == 0) *p.ticket = 0u;
    return;
  }
  // one warp per token: every lane keeps a sorted list of the best of its
  // keys (n = lane, lane + 32, ...); k rounds of a warp-wide argmax over the
  // list heads (key descending, lower id first) pick the winners in order
  for (int t = warp; t < T; t += kDecodeWarps) {
    TopK<16> tk;
    tk.init();
    const float* kt = kbuf + static_cast<size_t>(t) * N;
    const float* st = sbuf + static_cast<size_t>(t) * N;
    for (int base = 0; base < N; base += 32) {        // same trip count in every lane
      const int n = base + lane;
      const bool valid = n < N;
      tk.push_if(valid ? kt[n] : 0.0f, n, valid ? st[n] : 0.0f, valid);
    }
    float sum = 0.0f;
    int32_t* oid = p.out_ids + static_cast<size_t>(t) * p.k;
    float* ow = p.out_w + static_cast<size_t>(t) * p.k;
    for (int r = 0; r < p.k; ++r) {
      float bk = tk.key[0];
      int bi = tk.id[0];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xFFFFFFFFu, bk, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        if (topk_better(ok, oi, bk, bi)) { bk = ok; bi = oi; }
      }
      // the winning lane pops its head
      const bool mine = tk.id[0] == bi;
      const float bs = __shfl_sync(0xFFFFFFFFu, tk.sc[0], __ffs(__ballot_sync(0xFFFFFFFFu, mine)) - 1);
      if (mine) tk.pop_front();
      if (lane == 0) {
        oid[r] = bi;
        ow[r] = bs;                                            // the score, for now
        sum = __fadd_rn(sum, bs);
      }
    }
    if (lane == 0 && !p.raw) {
      for (int r = 0; r < p.k; ++r)
        ow[r] = sum > 0.0f ? __fdiv_rn(__fmul_rn(p.routed_scaling, ow[r]), sum) : 0.0f;
    }
  }
  if (tid == 0) *p.ticket = 0u;
}

// ------------------------------------------------------------------ host side

DecodePlan plan_decode(int64_t T, int64_t D, int64_t N, int num_sms, bool bf16) {
  DecodePlan d;
  if (T < 1 || T > 16 || N > 16384 || num_sms < 1) return d;
  d.tmax = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : T <= 8 ? 8 : 16;
  int epc = 1;
  while (epc < 8 && (N + epc - 1) / epc > num_sms) epc *= 2;
  // every thread prefetches at most kMaxBlocksPerThread weight blocks
  const int64_t gs = kDecodeThreads / epc;
  if ((D / kBlock + gs - 1) / gs > kMaxBlocksPerThread) return d;
  d.epc = epc;
  d.grid = static_cast<int>((N + epc - 1) / epc);
  // several tokens: clusters of CTAs share the staging and quantization of x
  // (the grid is padded to whole clusters; the extra CTAs have no experts)
  if (T >= 2 && d.grid >= kMaxDecodeCluster) {
    d.cluster = kMaxDecodeCluster;
    d.grid = (d.grid + kMaxDecodeCluster - 1) / kMaxDecodeCluster * kMaxDecodeCluster;
  }
  d.smem = decode_smem_layout(static_cast<int>(T), static_cast<int>(D), static_cast<int>(N), bf16 ? 2 : 4,
                              d.cluster).total;
  if (d.smem > kDecodeMaxSmem) return d;
  d.ok = true;
  return d;
}

template <bool kBF16>
static cudaError_t launch_t(const DecodeParams& p, const DecodePlan& plan, cudaStream_t s) {
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(decode_router_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kDecodeMaxSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // programmatic dependent launch (the kernel waits for its predecessor
  // before it reads anything but L2 prefetches), and for several tokens the
  // cluster
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = plan.cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = plan.cluster > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, decode_router_kernel<kBF16>, p);
}

cudaError_t launch_decode(const void* x, bool bf16, int64_t T, int64_t D, const uint8_t* W_codes,
                          const uint8_t* W_sf, const float* w_gsa, int64_t N, const float* bias,
                          int k, float routed_scaling, bool raw, int32_t* out_ids, float* out_w,
                          float* logits, float* ws_keys, float* ws_scores, uint32_t* ticket,
                          uint64_t* ws_words, uint32_t* status, bool test_stall, const DecodePlan& plan,
                          cudaStream_t s) {
  DecodeParams p;
  p.cluster = plan.cluster;
  p.x = x; p.T = static_cast<int>(T); p.D = static_cast<int>(D);
  p.W_codes = W_codes; p.W_sf = W_sf; p.w_gsa = w_gsa; p.N = static_cast<int>(N);
  p.bias = raw ? nullptr : bias; p.k = k; p.routed_scaling = routed_scaling;
  p.raw = raw ? 1 : 0; p.epc = plan.epc;
  p.out_ids = out_ids; p.out_w = out_w; p.logits = logits;
  p.ws_keys = ws_keys; p.ws_scores = ws_scores; p.ticket = ticket;
  p.ws_words = N <= 256 && T <= kMaxT ? ws_words : nullptr;
  p.status = status;
  p.test_stall = test_stall && p.ws_words ? 1 : 0;
  return bf16 ? launch_t<true>(p, plan, s) : launch_t<false>(p, plan, s);
}

}  // namespace nvr
