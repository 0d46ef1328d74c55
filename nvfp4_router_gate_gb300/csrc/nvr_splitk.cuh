// nvr_splitk.cuh -- pieces shared by the two K-split router GEMM kernels
// (gemm_splitk.cu: quantized x from the workspace; gemm_fused.cu: bf16 x
// quantized inside the GEMM): the TMA store of a CTA's fp32 partial logits
// and the tensor-map encoders.
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

}  // namespace nvr
