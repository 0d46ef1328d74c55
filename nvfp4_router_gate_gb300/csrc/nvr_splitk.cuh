// nvr_splitk.cuh -- pieces shared by the two K-split router GEMM kernels
// (gemm_splitk.cu: quantized x from the workspace; gemm_fused.cu: bf16 x
// quantized inside the GEMM): the stores of a CTA's fp32 partial logits, the
// tensor-map encoders and the per-token router epilogue.
#pragma once

#include "nvr_internal.h"
#include "nvr_tcgen05.cuh"

namespace nvr {

__device__ __forceinline__ uint4 ld_shared_v4(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)));
  return v;
}
__device__ __forceinline__ void st_shared_v4(uint8_t* p, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" :: "r"(smem_u32(p)), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Store this CTA's 128 x (128 * n_half) fp32 accumulator (tensor-memory
// columns 0..) to partial plane `rank`, rows m_tile*128.., with TMA.  Called by
// the eight warps 2-9: warp (quarter q = warp % 4, half h = (warp-2)/4) owns
// rows 32q..32q+31 and columns 128h..+127; each 32 x 32 block goes through one
// of the warp's two 4 KB staging buffers at stg_base + (warp-2) * 8 KB (128-byte
// swizzle, 1024-byte aligned).  `have_acc` false stores zeros.  Rows past T are
// not stored.  Returns after the stores have completed.
__device__ __forceinline__ void store_partial_tile(const CUtensorMap* tmap_p, uint8_t* stg_base, uint32_t tmem,
                                                   int warp, int lane, int m_tile, int rank, int n_half, int T,
                                                   bool have_acc) {
  const int q = warp & 3, h = (warp - 2) >> 2;
  if (h >= n_half || m_tile * 128 + q * 32 >= T) return;
  uint8_t* stg = stg_base + (warp - 2) * 8192;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    float v[32];
    if (have_acc) {
      tmem_load32(tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 128 + c * 32, v);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.0f;
    }
    uint8_t* buf = stg + (c & 1) * 4096;
    if (c >= 2) {
      if (lane == 0) bulk_wait_group_read<1>();
      __syncwarp();
    }
    // 128-byte swizzle: 16-byte chunk j of row r at chunk j ^ (r % 8)
#pragma unroll
    for (int j = 0; j < 8; ++j)
      st_shared_v4(buf + lane * 128 + ((j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tmap_p, buf, h * 128 + c * 32, m_tile * 128 + q * 32, rank);
      bulk_commit_group();
    }
    __syncwarp();
  }
  if (lane == 0) bulk_wait_group_all();
  __syncwarp();
}

// The fused router's accumulator into its partial plane, for a reader in
// another CTA of the same kernel (the tile's cluster or workspace barrier that
// follows makes the rows visible): of each row the n_groups groups of 128
// floats (tensor-memory columns 128 g .. for group g) are stored.  Called by the n_warps (8 or 16) warps from
// warp 2 on: warp w may only read tensor-memory lanes 32 (w % 4) .., so the
// n_warps / 4 warps of each lane quarter share its 4 n_groups blocks of
// 32 x 32 (block b: group b / 4, columns 32 (b % 4)).  Each block is staged
// (128-byte swizzle) in one of the warp's kBufs 4 KB buffers at
// stg_base + (warp-2) * kBufs * 4 KB (1024-byte aligned) and sent by TMA
// stores (tmap_p: encode_partial_rows) as two 16-row boxes -- a 112-row tile
// ends half-way through a lane quarter, and a 32-row box there would write
// the next tile's first rows; rows past T are clipped by the map.  Measured
// against coalesced stores from the warps (the same staging read back),
// prefill T = 4096: 39.8 against 40.0 us per call in graph replays (the CTAs'
// stores and tile barrier 0.3 us shorter).  Returns after the writes have
// completed (lane 0 waits for its bulk groups, then orders them before the
// generic proxy), so the caller's barrier publishes them like ordinary
// stores.  `have_acc` false stores zeros.
template <int kBufs>
__device__ __forceinline__ void store_partial_rows_tma(const CUtensorMap* tmap_p, uint8_t* stg_base, uint32_t tmem,
                                                       int warp, int lane, int row0, int rows, int rank,
                                                       int n_groups, bool have_acc, int n_warps) {
  const int w = warp - 2, q = warp & 3, j = w >> 2, wpq = n_warps >> 2;
  if (q * 32 >= rows) return;
  const int total = 4 * n_groups, per = (total + wpq - 1) / wpq;
  const int b_lo = j * per, b_hi = min(total, b_lo + per);
  if (b_lo >= b_hi) return;
  uint8_t* stg = stg_base + w * (kBufs * 4096);
  const bool second = q * 32 + 16 < rows;
  int n = 0;
#pragma unroll 1
  for (int blk = b_lo; blk < b_hi; ++blk, ++n) {
    const int col0 = (blk >> 2) * 128 + (blk & 3) * 32;
    float v[32];
    if (have_acc) {
      tmem_load32(tmem + (static_cast<uint32_t>(q * 32) << 16) + col0, v);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.0f;
    }
    uint8_t* buf = stg + (n % kBufs) * 4096;
    if (n >= kBufs) {                                // the buffer's previous block has been read
      if (lane == 0) bulk_wait_group_read<kBufs - 1>();
      __syncwarp();
    }
#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
      st_shared_v4(buf + lane * 128 + ((jj ^ (lane & 7)) << 4), v[4 * jj], v[4 * jj + 1], v[4 * jj + 2],
                   v[4 * jj + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tmap_p, buf, col0, row0 + q * 32, rank);
      if (second) tma_store_3d(tmap_p, buf + 2048, col0, row0 + q * 32 + 16, rank);
      bulk_commit_group();
    }
    __syncwarp();
  }
  if (lane == 0) {
    bulk_wait_group_all();
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  __syncwarp();
}

// Packed-code operand [rows, D/2] uint8 read in boxes of 128 bytes x box_rows,
// 128-byte swizzle.
inline bool encode_codes(CUtensorMap* map, const uint8_t* ptr, int64_t rows, int64_t D, uint32_t box_rows) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D / 2), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D / 2)};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(ptr), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Partial rows [S][T][row_floats] fp32 of the fused router, stored in boxes of
// 32 floats x 16 rows with 128-byte swizzle (store_partial_rows_tma).
inline bool encode_partial_rows(CUtensorMap* map, float* ptr, int64_t T, int S, int row_floats) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(row_floats), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(S)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_floats) * 4, static_cast<cuuint64_t>(T) * row_floats * 4};
  cuuint32_t box[3] = {32, 16, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Partial logits [S][T][256] fp32, stored in 32 x 32 boxes with 128-byte swizzle.
inline bool encode_partials(CUtensorMap* map, float* ptr, int64_t T, int S) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  cuuint64_t dims[3] = {256, static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(S)};
  cuuint64_t strides[2] = {256 * 4, static_cast<cuuint64_t>(T) * 256 * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------ router epilogue
//
// One warp routes one token from its S fp32 partial-logit rows (row stride
// 128 NG floats, planes `plane` floats apart), NG = 2 for heads of up to 256
// experts, 3 for up to 384: lane l owns experts 128 g + 4l .. 128 g + 4l + 3
// of every group g (coalesced 512-byte rows).  The partials are added in
// rank order (the result does not depend on timing), scaled by
// gsa_x * gsa_w; keys are sigmoid(logit) + bias (RAW: the logit).
// Selection, on (key, id) pairs packed into order-preserving 64-bit words:
// - sorted lists: each lane sorts its words of groups 0-1 (8) and, with
//   NG = 3, those of group 2 in a second list of 4; k rounds take the best
//   head of the warp (two 32-bit max reductions: the key's bits, then the
//   complemented id among the lanes holding that key) and the winning lane
//   pops it;
// - rank selection (NG = 2): the k-th largest of the 32 lanes' maxima of the
//   key bits (ranked by counting, one reduction) bounds the k-th best key
//   from below, the words at or above it (typically k to 2k) are gathered
//   into one list by ballots, and each candidate's rank among them -- a
//   count of better candidates -- is its rank overall; with more than 32
//   candidates (many equal keys) the bound is taken again on whole words,
//   else the sorted lists select.
// Both exact for any keys, ties included (equal keys: lower id first).  The
// selected experts' logits come back from the warp's copy of the row in
// shared memory; the weights are routed_scaling * score / (sum of the k
// scores).

// (key descending, id ascending) as one unsigned 64-bit order: the float's
// order-preserving bit pattern above the complemented id.  Never 0 for a
// non-NaN key, so 0 marks "no entry".
__device__ __forceinline__ uint64_t pack_key(float key, int id) {
  const uint32_t b = __float_as_uint(key);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(id));
}

// Compare-exchange so that v[a] >= v[b]; the 19-comparator 8-sorter (the
// network of sort8 in nvr_device.cuh) and the 5-comparator 4-sorter on packed
// keys.
template <int M>
__device__ __forceinline__ void cx(uint64_t (&v)[M], int a, int b) {
  const uint64_t x = v[a], y = v[b];
  const bool sw = y > x;
  v[a] = sw ? y : x;
  v[b] = sw ? x : y;
}
__device__ __forceinline__ void sort8_desc(uint64_t (&v)[8]) {
  cx(v, 0, 2); cx(v, 1, 3); cx(v, 4, 6); cx(v, 5, 7);
  cx(v, 0, 4); cx(v, 1, 5); cx(v, 2, 6); cx(v, 3, 7);
  cx(v, 0, 1); cx(v, 2, 3); cx(v, 4, 5); cx(v, 6, 7);
  cx(v, 2, 4); cx(v, 3, 5);
  cx(v, 1, 4); cx(v, 3, 6);
  cx(v, 1, 2); cx(v, 3, 4); cx(v, 5, 6);
}
__device__ __forceinline__ void sort4_desc(uint64_t (&v)[4]) {
  cx(v, 0, 1); cx(v, 2, 3);
  cx(v, 0, 2); cx(v, 1, 3);
  cx(v, 1, 2);
}

// Shared memory of one token slot of a router warp, in float4: the token's
// 128 NG logits.
template <int NG>
struct RouteSlot {
  static constexpr int kFloat4 = 32 * NG;
};
constexpr int kRouteSlot = RouteSlot<2>::kFloat4;
// Shared memory of one token slot's selection: 32 lane maxima, up to 32
// candidate words and the k <= 16 selected ids.
constexpr int kRouteScratch = 32 * 4 + 32 * 8 + 16 * 4;

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}

// Rank selection of the k best of a warp's words (at most 32 candidates at
// or above `bound`, gathered into s_c by ballots) -- the candidates' ranks
// among themselves are their ranks overall; returns false (s_sel untouched)
// when more than 32 words reach the bound.
template <int kE>
__device__ __forceinline__ bool select_by_rank(const uint64_t (&pw)[kE], uint64_t bound, int k, int lane,
                                               uint64_t* s_c, int* s_sel) {
  const uint32_t lt = (1u << lane) - 1u;
  int base = 0;
#pragma unroll
  for (int j = 0; j < kE; ++j) {
    const bool c = pw[j] != 0 && pw[j] >= bound;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, c);
    const int pos = base + __popc(bal & lt);
    if (c && pos < 32) s_c[pos] = pw[j];
    base += __popc(bal);
  }
  if (base > 32) return false;
  __syncwarp();
  if (lane < base) {
    const uint64_t me = s_c[lane];
    int rk = 0;
#pragma unroll 4
    for (int q = 0; q < base; ++q) rk += s_c[q] > me ? 1 : 0;
    if (rk < k) s_sel[rk] = static_cast<int>(~static_cast<uint32_t>(me));
  }
  return true;
}

// The k best of a warp's words when many share their key bits: the k-th
// largest lane maximum of the whole words bounds them (exact ties then leave
// the lowest ids, about 4k words); past 32 candidates each lane sorts its
// words and k rounds take the best head of the warp (two 32-bit max
// reductions: the key's bits, then the complemented id among the lanes
// holding that key), the winning lane popping it.
template <int kE>
__device__ __forceinline__ void select_ties(uint64_t (&pw)[kE], int k, int lane, uint64_t* s_c, int* s_sel) {
  uint64_t m = 0;
#pragma unroll
  for (int j = 0; j < kE; ++j) m = pw[j] > m ? pw[j] : m;
  __syncwarp();
  s_c[lane] = m;
  __syncwarp();
  int rk = 0;
#pragma unroll 8
  for (int q = 0; q < 32; ++q) rk += s_c[q] > m ? 1 : 0;
  __syncwarp();
  const uint64_t v = rk < k ? m : ~0ull;
  const uint32_t hmin = __reduce_min_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32));
  const uint32_t lmin = __reduce_min_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32) == hmin
                                                           ? static_cast<uint32_t>(v) : 0xFFFFFFFFu);
  if (select_by_rank(pw, (static_cast<uint64_t>(hmin) << 32) | lmin, k, lane, s_c, s_sel)) return;
  constexpr int kB = kE > 8 ? kE - 8 : 1;
  uint64_t pa[8], pb[kB];
#pragma unroll
  for (int j = 0; j < 8; ++j) pa[j] = pw[j];
#pragma unroll
  for (int j = 0; j < kB; ++j) pb[j] = kE > 8 ? pw[8 + j] : 0;
  sort8_desc(pa);
  if constexpr (kB == 4) sort4_desc(pb);
#pragma unroll 1
  for (int r = 0; r < k; ++r) {
    const bool from_b = kE > 8 && pb[0] > pa[0];
    const uint64_t h = from_b ? pb[0] : pa[0];
    const uint32_t hi = static_cast<uint32_t>(h >> 32), lo = static_cast<uint32_t>(h);
    const uint32_t hmax = __reduce_max_sync(0xFFFFFFFFu, hi);
    const uint32_t lmax = __reduce_max_sync(0xFFFFFFFFu, hi == hmax ? lo : 0u);
    const bool win = hi == hmax && lo == lmax;                 // ids are unique
    const bool wa = win && !from_b, wb = win && from_b;
#pragma unroll
    for (int j = 0; j < 7; ++j) pa[j] = wa ? pa[j + 1] : pa[j];
    pa[7] = wa ? 0 : pa[7];
#pragma unroll
    for (int j = 0; j + 1 < kB; ++j) pb[j] = wb ? pb[j + 1] : pb[j];
    pb[kB - 1] = wb ? 0 : pb[kB - 1];
    if (lane == 0) s_sel[r] = static_cast<int>(~lmax);
  }
}

template <int NG>
struct TokenRouterT {
  static_assert(NG == 2 || NG == 3, "heads of up to 256 or 384 experts");
  static constexpr int kE = 4 * NG;        // experts per lane
  static constexpr int kRow = 128 * NG;    // floats per partial row
  float b[kE];                 // bias of this lane's experts (0 in RAW mode or without bias)
  int N, k, raw;
  float routed_scaling;

  __device__ __forceinline__ static int col_of(int j, int lane) { return 128 * (j >> 2) + 4 * lane + (j & 3); }

  // The bias is a caller input that no kernel of the call writes; the call's
  // first kernel has already waited for the caller's previous kernel (which
  // may have written it), so a later kernel of the call may read it before
  // its own grid-dependency wait.
  __device__ __forceinline__ void init(const float* bias, int N_, int k_, int raw_, float rs, int lane) {
    N = N_; k = k_; raw = raw_; routed_scaling = rs;
#pragma unroll
    for (int j = 0; j < kE; ++j) {
      const int col = col_of(j, lane);
      b[j] = (!raw && bias && col < N) ? __ldg(bias + col) : 0.0f;
    }
  }

  // Routes NT tokens at once (independent dependency chains interleave);
  // t[i] < 0 marks an unused slot.  s_row: NT token slots of
  // RouteSlot<NG>::kFloat4 float4 for the warp.  kRank (up to 256 experts):
  // the rank selection, with scratch = NT x kRouteScratch bytes (16-byte
  // aligned) of the warp's selection lists; else the sorted lists and k
  // rounds of a warp arg-max.  (Measured: the rank selection shortens the
  // separate epilogue kernel, one token per warp, by ~0.9 us at T = 4096;
  // inside the fused kernel its code and registers cost as much as it saves.)  stage: null, or shared
  // memory for the warp's partial rows (row n * S + s: 32 NG float4 of token
  // slot n, plane s; only the rows of valid slots are touched) -- then every
  // partial row is copied in at once (asynchronous copies, one round trip to
  // L2 whatever S) before the sums.
  template <int NT, bool kRank = false>
  __device__ __forceinline__ void route(const float* partials, size_t plane, int S, const int64_t (&t)[NT],
                                        float gscale, float4* s_row, int lane, int32_t* out_ids, float* out_w,
                                        float* logits, float4* stage = nullptr, uint8_t* scratch = nullptr) const {
    constexpr int kSlot = RouteSlot<NG>::kFloat4;
    float4 a[NT][NG];
    if (stage) {
      for (int s = 0; s < S; ++s)
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          if (t[n] < 0) continue;
          const float* r = partials + static_cast<size_t>(t[n]) * kRow + s * plane;
          float4* d = stage + kSlot * (n * S + s);
#pragma unroll
          for (int g = 0; g < NG; ++g)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(d + 32 * g + lane)),
                         "l"(reinterpret_cast<uint64_t>(r + 128 * g + 4 * lane)) : "memory");
        }
      asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
      // each lane reads back only what it copied itself: no warp barrier needed
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const bool ok = t[n] >= 0;
#pragma unroll
        for (int g = 0; g < NG; ++g)
          a[n][g] = ok ? stage[kSlot * (n * S) + 32 * g + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int s = 1; s < S; ++s)                        // partials in rank order
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          if (t[n] < 0) continue;
#pragma unroll
          for (int g = 0; g < NG; ++g) a[n][g] = add4(a[n][g], stage[kSlot * (n * S + s) + 32 * g + lane]);
        }
    } else {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const float* row = partials + static_cast<size_t>(t[n] < 0 ? 0 : t[n]) * kRow;
#pragma unroll
        for (int g = 0; g < NG; ++g) a[n][g] = __ldcg(reinterpret_cast<const float4*>(row + 128 * g + 4 * lane));
      }
#pragma unroll 2
      for (int s = 1; s < S; ++s) {                      // partials in rank order
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const float* r = partials + static_cast<size_t>(t[n] < 0 ? 0 : t[n]) * kRow + s * plane;
#pragma unroll
          for (int g = 0; g < NG; ++g)
            a[n][g] = add4(a[n][g], __ldcg(reinterpret_cast<const float4*>(r + 128 * g + 4 * lane)));
        }
      }
    }
    float l[NT][kE];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        l[n][4 * g] = __fmul_rn(a[n][g].x, gscale);
        l[n][4 * g + 1] = __fmul_rn(a[n][g].y, gscale);
        l[n][4 * g + 2] = __fmul_rn(a[n][g].z, gscale);
        l[n][4 * g + 3] = __fmul_rn(a[n][g].w, gscale);
      }
    if (logits) {
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int j = 0; j < kE; ++j)
          if (t[n] >= 0 && col_of(j, lane) < N) logits[t[n] * N + col_of(j, lane)] = l[n][j];
      return;
    }
    int sel_id[NT];
    if constexpr (!kRank || NG == 3) {
      // the lanes' sorted lists and k rounds of a warp arg-max
      // lists: groups 0-1 (8 words), and group 2 (4 words) when NG = 3
      constexpr int kB = NG == 3 ? 4 : 1;
      uint64_t pa[NT][8], pb[NT][kB];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int g = 0; g < NG; ++g)
          s_row[kSlot * n + 32 * g + lane] = make_float4(l[n][4 * g], l[n][4 * g + 1], l[n][4 * g + 2], l[n][4 * g + 3]);
#pragma unroll
        for (int j = 0; j < kE; ++j) {
          const float key = raw ? l[n][j] : __fadd_rn(sigmoid_f32(l[n][j]), b[j]);
          const uint64_t w = col_of(j, lane) < N ? pack_key(key, col_of(j, lane)) : 0;
          if (j < 8) pa[n][j] = w;
          else pb[n][(j - 8) & (kB - 1)] = w;
        }
        sort8_desc(pa[n]);
        if constexpr (NG == 3) sort4_desc(pb[n]);
        else pb[n][0] = 0;
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) sel_id[n] = 0;
      // Each reduction takes ~90 cycles and issue is in order: the NT tokens'
      // reductions of a round are issued back to back so their latencies overlap.
#pragma unroll 1
      for (int r = 0; r < k; ++r) {
        uint32_t hi[NT], lo[NT], hmax[NT], lmax[NT];
        bool from_b[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          from_b[n] = NG == 3 && pb[n][0] > pa[n][0];
          const uint64_t h = from_b[n] ? pb[n][0] : pa[n][0];
          hi[n] = static_cast<uint32_t>(h >> 32);
          lo[n] = static_cast<uint32_t>(h);
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) hmax[n] = __reduce_max_sync(0xFFFFFFFFu, hi[n]);
#pragma unroll
        for (int n = 0; n < NT; ++n) lmax[n] = __reduce_max_sync(0xFFFFFFFFu, hi[n] == hmax[n] ? lo[n] : 0u);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          if (lane == r) sel_id[n] = static_cast<int>(~lmax[n]);   // the winning expert
          const bool win = hi[n] == hmax[n] && lo[n] == lmax[n];     // its lane (ids are unique)
          const bool wa = win && !from_b[n], wb = win && from_b[n];
#pragma unroll
          for (int j = 0; j < 7; ++j) pa[n][j] = wa ? pa[n][j + 1] : pa[n][j];
          pa[n][7] = wa ? 0 : pa[n][7];
          if constexpr (NG == 3) {
#pragma unroll
            for (int j = 0; j < 3; ++j) pb[n][j] = wb ? pb[n][j + 1] : pb[n][j];
            pb[n][3] = wb ? 0 : pb[n][3];
          }
        }
      }
      __syncwarp();
    } else {
      // (key, id) words of this lane's experts (0: no expert)
      uint64_t pw[NT][kE];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int g = 0; g < NG; ++g)
          s_row[kSlot * n + 32 * g + lane] = make_float4(l[n][4 * g], l[n][4 * g + 1], l[n][4 * g + 2], l[n][4 * g + 3]);
#pragma unroll
        for (int j = 0; j < kE; ++j) {
          const float key = raw ? l[n][j] : __fadd_rn(sigmoid_f32(l[n][j]), b[j]);
          pw[n][j] = col_of(j, lane) < N ? pack_key(key, col_of(j, lane)) : 0;
        }
      }
      // A lower bound of the k-th best key: the k-th largest of the 32 lanes'
      // maxima of the key bits (the k largest maxima are k keys at least that
      // large), found as the least maximum whose rank among the maxima (count
      // of larger ones) is below k.
      uint32_t* s_m = reinterpret_cast<uint32_t*>(scratch);                        // [NT][32]
      uint64_t* s_c = reinterpret_cast<uint64_t*>(scratch + NT * 128);              // [NT][32]
      int* s_sel = reinterpret_cast<int*>(scratch + NT * 384);                      // [NT][16]
      uint32_t bound[NT];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < kE; ++j) m = max(m, static_cast<uint32_t>(pw[n][j] >> 32));
        bound[n] = m;
        s_m[32 * n + lane] = m;
      }
      __syncwarp();
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        int rk = 0;
        const uint4* q4 = reinterpret_cast<const uint4*>(s_m + 32 * n);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 v = q4[q];
          rk += (v.x > bound[n]) + (v.y > bound[n]) + (v.z > bound[n]) + (v.w > bound[n]);
        }
        bound[n] = rk < k ? bound[n] : 0xFFFFFFFFu;
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) bound[n] = __reduce_min_sync(0xFFFFFFFFu, bound[n]);
      // Candidates: the words whose key bits reach the bound (the k best are
      // among them), packed into the slot's list by per-expert ballots.
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        sel_id[n] = 0;
        if (!select_by_rank(pw[n], static_cast<uint64_t>(bound[n]) << 32, k, lane, s_c + 32 * n, s_sel + 16 * n)) {
          // many equal key bits: the bound again on whole words (the id breaks
          // the ties, so exact ties leave about 4k candidates), else sorted
          // lists and k rounds of a warp arg-max
          select_ties(pw[n], k, lane, s_c + 32 * n, s_sel + 16 * n);
        }
      }
      __syncwarp();
#pragma unroll
      for (int n = 0; n < NT; ++n) sel_id[n] = lane < k ? s_sel[16 * n + lane] : 0;
      __syncwarp();
    }
    const bool mine = lane < k;
    float sc[NT], sum[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int id = sel_id[n];
      const float sel_l = reinterpret_cast<const float*>(s_row + kSlot * n)[(id >= 0 && id < kRow) ? id : 0];
      sc[n] = raw ? sel_l : sigmoid_f32(sel_l);
      sum[n] = mine ? sc[n] : 0.0f;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int n = 0; n < NT; ++n) sum[n] = __fadd_rn(sum[n], __shfl_xor_sync(0xFFFFFFFFu, sum[n], o));
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      if (mine && t[n] >= 0) {
        float w = sc[n];
        if (!raw) w = sum[n] > 0.0f ? __fdiv_rn(__fmul_rn(routed_scaling, sc[n]), sum[n]) : 0.0f;
        out_ids[t[n] * k + lane] = sel_id[n];
        out_w[t[n] * k + lane] = w;
      }
    }
    __syncwarp();                                      // s_row is reused by the warp's next tokens
  }
};

using TokenRouter = TokenRouterT<2>;

}  // namespace nvr
