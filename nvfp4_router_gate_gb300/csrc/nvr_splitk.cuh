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

// The same tile with ordinary stores, for a reader in another CTA of the
// same kernel (the tile's cluster or workspace barrier that follows makes them
// visible): each 32 x 32 block goes through the warp's 4 KB staging buffer at
// stg_base + (warp-2) * 4 KB (128-byte swizzle, conflict-free both ways) and
// leaves as 512-byte coalesced rows.  Called by n_warps = 8 or 16 warps from
// warp 2 on; with 16, warps 2-9 store column blocks 0-1 of their quarter and
// half, warps 10-17 blocks 2-3.
__device__ __forceinline__ void store_partial_rows(float* plane, uint8_t* stg_base, uint32_t tmem, int warp,
                                                   int lane, int64_t row0, int rows, int n_half, bool have_acc,
                                                   int n_warps = 8) {
  const int w = warp - 2, q = warp & 3, h = (w >> 2) & 1;
  if (h >= n_half || q * 32 >= rows) return;
  const int c_lo = n_warps == 16 ? 2 * (w >> 3) : 0, c_hi = n_warps == 16 ? c_lo + 2 : 4;
  uint8_t* buf = stg_base + w * 4096;
#pragma unroll 1
  for (int c = c_lo; c < c_hi; ++c) {
    float v[32];
    if (have_acc) {
      tmem_load32(tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 128 + c * 32, v);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      st_shared_v4(buf + lane * 128 + ((j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 4 * i + (lane >> 3), j = lane & 7;
      const uint4 val = ld_shared_v4(buf + r * 128 + ((j ^ (r & 7)) << 4));
      if (q * 32 + r < rows)
        *reinterpret_cast<uint4*>(plane + (row0 + q * 32 + r) * 256 + h * 128 + c * 32 + 4 * j) = val;
    }
    __syncwarp();
  }
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
// One warp routes one token from its S fp32 partial-logit rows (planes
// `plane` floats apart): lane l owns experts 4l..4l+3 and 128+4l..128+4l+3
// (coalesced 512-byte rows).  The partials are added in rank order (the
// result does not depend on timing), scaled by gsa_x * gsa_w; keys are
// sigmoid(logit) + bias (RAW: the logit).  Selection: each lane sorts its 8
// (key, id) pairs packed into order-preserving 64-bit words; k rounds then
// take the best head of the warp (two 32-bit max reductions: the key's bits,
// then the complemented id among the lanes holding that key) and the winning
// lane pops its head.  Exact for any keys, ties included (equal keys: lower
// id first), with no data-dependent trip counts.  The selected experts'
// logits come back from the warp's copy of the row in shared memory; the
// weights are routed_scaling * score / (sum of the k scores).

// (key descending, id ascending) as one unsigned 64-bit order: the float's
// order-preserving bit pattern above the complemented id.  Never 0 for a
// non-NaN key, so 0 marks "no entry".
__device__ __forceinline__ uint64_t pack_key(float key, int id) {
  const uint32_t b = __float_as_uint(key);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(id));
}

// Compare-exchange so that v[a] >= v[b]; the 19-comparator 8-sorter (the
// network of sort8 in nvr_device.cuh) on packed keys.
__device__ __forceinline__ void cx(uint64_t (&v)[8], int a, int b) {
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

// Shared memory of one token slot of a router warp, in float4: the token's
// 256 logits.
constexpr int kRouteSlot = 64;

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}

struct TokenRouter {
  float b[8];                  // bias of this lane's experts (0 in RAW mode or without bias)
  int N, k, raw;
  float routed_scaling;

  // The bias is a caller input that no kernel of the call writes; the call's
  // first kernel has already waited for the caller's previous kernel (which
  // may have written it), so a later kernel of the call may read it before
  // its own grid-dependency wait.
  __device__ __forceinline__ void init(const float* bias, int N_, int k_, int raw_, float rs, int lane) {
    N = N_; k = k_; raw = raw_; routed_scaling = rs;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int col = (j < 4 ? 0 : 128) + 4 * lane + (j & 3);
      b[j] = (!raw && bias && col < N) ? __ldg(bias + col) : 0.0f;
    }
  }

  // Routes NT tokens at once (independent dependency chains interleave);
  // t[i] < 0 marks an unused slot.  s_row: NT rows of 64 float4 for the warp.
  // stage: null, or shared memory for the warp's partial rows (row n * S + s:
  // 64 float4 of token slot n, plane s; only the rows of valid slots are
  // touched) -- then every partial row is copied in at once (asynchronous
  // copies, one round trip to L2 whatever S) before the sums.
  template <int NT>
  __device__ __forceinline__ void route(const float* partials, size_t plane, int S, const int64_t (&t)[NT],
                                        float gscale, float4* s_row, int lane, int32_t* out_ids, float* out_w,
                                        float* logits, float4* stage = nullptr) const {
    float4 a0[NT], a1[NT];
    if (stage) {
      for (int s = 0; s < S; ++s)
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          if (t[n] < 0) continue;
          const float* r = partials + static_cast<size_t>(t[n]) * 256 + s * plane;
          float4* d = stage + 64 * (n * S + s);
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(d + lane)),
                       "l"(reinterpret_cast<uint64_t>(r + 4 * lane)) : "memory");
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(d + 32 + lane)),
                       "l"(reinterpret_cast<uint64_t>(r + 128 + 4 * lane)) : "memory");
        }
      asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
      // each lane reads back only what it copied itself: no warp barrier needed
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const bool ok = t[n] >= 0;
        a0[n] = ok ? stage[64 * (n * S) + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        a1[n] = ok ? stage[64 * (n * S) + 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int s = 1; s < S; ++s)                        // partials in rank order
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          if (t[n] < 0) continue;
          a0[n] = add4(a0[n], stage[64 * (n * S + s) + lane]);
          a1[n] = add4(a1[n], stage[64 * (n * S + s) + 32 + lane]);
        }
    } else {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const float* row = partials + static_cast<size_t>(t[n] < 0 ? 0 : t[n]) * 256;
        a0[n] = __ldcg(reinterpret_cast<const float4*>(row + 4 * lane));
        a1[n] = __ldcg(reinterpret_cast<const float4*>(row + 128 + 4 * lane));
      }
#pragma unroll 2
      for (int s = 1; s < S; ++s) {                      // partials in rank order
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const float* r = partials + static_cast<size_t>(t[n] < 0 ? 0 : t[n]) * 256 + s * plane;
          a0[n] = add4(a0[n], __ldcg(reinterpret_cast<const float4*>(r + 4 * lane)));
          a1[n] = add4(a1[n], __ldcg(reinterpret_cast<const float4*>(r + 128 + 4 * lane)));
        }
      }
    }
    int col[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) col[j] = (j < 4 ? 0 : 128) + 4 * lane + (j & 3);
    float l[NT][8];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const float acc[8] = {a0[n].x, a0[n].y, a0[n].z, a0[n].w, a1[n].x, a1[n].y, a1[n].z, a1[n].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) l[n][j] = __fmul_rn(acc[j], gscale);
    }
    if (logits) {
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (t[n] >= 0 && col[j] < N) logits[t[n] * N + col[j]] = l[n][j];
      return;
    }
    uint64_t pk[NT][8];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      s_row[64 * n + lane] = make_float4(l[n][0], l[n][1], l[n][2], l[n][3]);
      s_row[64 * n + 32 + lane] = make_float4(l[n][4], l[n][5], l[n][6], l[n][7]);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float key = raw ? l[n][j] : __fadd_rn(sigmoid_f32(l[n][j]), b[j]);
        pk[n][j] = col[j] < N ? pack_key(key, col[j]) : 0;
      }
      sort8_desc(pk[n]);
    }
    int sel_id[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) sel_id[n] = 0;
    // Each reduction takes ~90 cycles and issue is in order: the NT tokens'
    // reductions of a round are issued back to back so their latencies overlap.
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
      uint32_t hi[NT], lo[NT], hmax[NT], lmax[NT];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        hi[n] = static_cast<uint32_t>(pk[n][0] >> 32);
        lo[n] = static_cast<uint32_t>(pk[n][0]);
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) hmax[n] = __reduce_max_sync(0xFFFFFFFFu, hi[n]);
#pragma unroll
      for (int n = 0; n < NT; ++n) lmax[n] = __reduce_max_sync(0xFFFFFFFFu, hi[n] == hmax[n] ? lo[n] : 0u);
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        if (lane == r) sel_id[n] = static_cast<int>(~lmax[n]);   // the winning expert
        const bool win = hi[n] == hmax[n] && lo[n] == lmax[n];     // its lane (ids are unique)
#pragma unroll
        for (int j = 0; j < 7; ++j) pk[n][j] = win ? pk[n][j + 1] : pk[n][j];
        pk[n][7] = win ? 0 : pk[n][7];
      }
    }
    __syncwarp();
    const bool mine = lane < k;
    float sc[NT], sum[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const float sel_l = reinterpret_cast<const float*>(s_row + 64 * n)[sel_id[n] & 255];
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

}  // namespace nvr
