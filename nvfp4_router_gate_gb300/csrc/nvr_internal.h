// nvr_internal.h -- host-side declarations shared by the router's .cu files:
// launch configurations, the workspace layout and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/nvfp4_router.h"
#include "nvr_device.cuh"

namespace nvr {

constexpr int kAmaxThreads = 256;
constexpr int kQuantThreads = 256;
constexpr int kMaxAmaxGrid = 4096;       // partial slots in the workspace
constexpr int kMaxSplits = 256;          // N splits per M tile (bounds the workspace)
constexpr int kMaxKmax = 16;             // largest top-k list
constexpr int kMaxDevices = 64;
constexpr int kMaxTicketTiles = 65536;   // token tiles of the N-split router (T <= 8,388,608)
constexpr int kMaxFlatTiles = 1024;      // token tiles of a fused router launched without clusters
constexpr int kDecodeWords = 16 * 256;   // decode collector words: up to 16 tokens x 256 experts

// cuTensorMapEncodeTiled, fetched from the driver through the runtime (no
// link-time dependency on libcuda).
typedef CUresult (*TensorMapEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                      const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                      const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                      CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
TensorMapEncodeFn tensor_map_encoder();

// Number of SMs of the current device (cached per device); 0 on error.
int device_sm_count();

// NVR_OK for cudaSuccess, else NVR_ERR_CUDA; records the error for
// nvr_last_cuda_error (per host thread).
nvr_status cuda_status(cudaError_t e);

struct GemmPlan {
  int m_tiles = 0, n_tiles = 0, n_splits = 1;
};
GemmPlan plan_gemm(int64_t T, int64_t N, int num_sms);

// Decode (single-launch) path limits and plan.  A decode CTA's shared memory
// (at most kDecodeMaxSmem) holds the keys and scores of every (token, expert)
// pair, T * N * 8 bytes, so a shape the plan accepts never needs more scratch
// for them than that.
constexpr int kDecodeMaxSmem = 224 * 1024;
struct DecodePlan {
  bool ok = false;
  int tmax = 0;        // template bucket >= T
  int epc = 0;         // experts per CTA
  int grid = 0;
  int cluster = 1;     // CTAs per cluster sharing the staging and quantization of x
  size_t smem = 0;
};
DecodePlan plan_decode(int64_t T, int64_t D, int64_t N, int num_sms, bool bf16);

// Byte offsets inside the caller's workspace.
struct WsLayout {
  size_t control = 0;        // 256 bytes: status word and tickets
  size_t amax_partials = 0;  // kMaxAmaxGrid x u32
  size_t scalars = 0;        // x gsa (router path), quantizer record {gsa, 1/gsa, mode, amax} -- 256 bytes
  size_t tickets = 0;        // kMaxTicketTiles x u32: the N-split router's per-tile tickets
  size_t tile_sync = 0;      // 2 x kMaxFlatTiles u32: the fused router's tile-barrier counters (no clusters)
  size_t dec_words = 0;      // kDecodeWords u64: the decode collector's (key, score) words, zero between calls
  size_t x_codes = 0;        // [rows_pad, D/2]
  size_t x_sf = 0;           // tile layout, rows_pad rows
  size_t partials = 0;       // N-split top-k lists, or the K-split fp32 partial logits
  size_t decode = 0;         // decode scratch: keys and scores [T, N] fp32
  size_t total = 0;
};
WsLayout router_ws_layout(int64_t T, int64_t D, int64_t N);
WsLayout quantize_ws_layout(int64_t rows, int64_t D);

// ----------------------------------------------------------------- launchers
cudaError_t launch_amax(const void* x, bool bf16, int64_t n_elems, uint32_t* partials,
                        uint32_t* ticket, float* gsa_out, float* qrec, int grid,
                        cudaStream_t s);
cudaError_t launch_amax_bulk(const void* x, bool bf16, int64_t n_elems, uint32_t* partials,
                             uint32_t* ticket, float* gsa_out, float* qrec, uint32_t* status,
                             int grid, cudaStream_t s);
cudaError_t launch_quantize(const void* x, bool bf16, int64_t rows, int64_t D, bool tiled,
                            const float* qrec, uint8_t* codes, uint8_t* sf, cudaStream_t s);
int amax_grid(int64_t n_elems, bool bf16, int num_sms);

nvr_status launch_gemm_topk(const uint8_t* x_codes, const uint8_t* x_sf, const float* x_gsa,
                            int64_t T, int64_t D, const uint8_t* W_codes, const uint8_t* W_sf,
                            const float* w_gsa, int64_t N, const float* bias, int k,
                            float routed_scaling, bool raw, int32_t* out_ids, float* out_w,
                            void* logits, bool logits_bf16, float4* partials, uint32_t* tickets,
                            uint32_t* status, const GemmPlan& g, bool test_stall, cudaStream_t s);

// Few tokens (T <= 128), many outputs: the weight-streaming GEMM with the
// token tile as the MMA's N (32, 64 or 128 columns), n_splits CTAs over the
// 128-row weight tiles.  Top-k mode (out == null): per-token candidates
// merged by the last CTA (partials: [128][n_splits * k] float4; tickets: the
// ticket at word 0, per-token counts at words 64..191, per-token 32 64-bit
// slot words at words 512..8703, all left at zero); logits mode: out [T, N] fp32
// or bf16.  stream_splits: CTAs for N outputs.
int stream_token_tile(int64_t T);
int stream_splits(int64_t N, int num_sms);
nvr_status launch_gemm_stream(const uint8_t* x_codes, const uint8_t* x_sf, const float* x_gsa, int64_t T, int64_t D,
                              const uint8_t* W_codes, const uint8_t* W_sf, const float* w_gsa, int64_t N,
                              const float* bias, int k, float routed_scaling, bool raw, int32_t* out_ids,
                              float* out_w, void* out, bool out_bf16, float4* partials, uint32_t* ticket,
                              uint32_t* status, int n_splits, bool test_stall, cudaStream_t s);

// Router for N <= 256: the GEMM split along K over S CTAs (fp32 partials in
// the workspace), then the warp-per-token epilogue kernel.
// splitk_partial_rows(T): rows (of 256 fp32; 384 for the fused kernel's
// 257-384-expert heads, whose partial region is sized accordingly) the partial region holds for T
// tokens, an upper bound of S * T_pad for every S plan_splitk picks on a GPU
// with at most 256 SMs; plan_splitk: S for T tokens.
constexpr int kMaxSplitK = 16;
size_t splitk_partial_rows(int64_t T);
int plan_splitk(int64_t T, int64_t D, int num_sms);
nvr_status launch_splitk_gemm(const uint8_t* x_codes, const uint8_t* x_sf, int64_t T, int64_t D,
                              const uint8_t* W_codes, const uint8_t* W_sf, int64_t N, float* partials,
                              uint32_t* status, int S, bool test_stall, cudaStream_t s);
// The router for bf16 activations and N <= 384 in one kernel: quantization
// inside the K-split GEMM, partials through L2 and the epilogue (S CTAs per
// token tile of tile_rows = 128 or 112 rows, S in {1,2,4,8,16}).  With
// amax_sync (5 zeroed workspace words) the kernel also computes max|x| itself
// and publishes qrec and x_gsa -- every CTA of the grid must then be resident
// at once; without it, qrec and x_gsa come from the amax kernel launched
// before.  tile_sync (2 x kMaxFlatTiles zeroed workspace words) comes with
// amax_sync.  flat (needs amax_sync): the launch has no clusters and a tile's
// CTAs meet at a workspace barrier -- the grid must then be resident at once;
// else each tile's CTAs form a cluster.
// fused_cluster_capacity(S): clusters of S CTAs the device holds at once;
// fused_block_capacity(): CTAs it holds at once without clusters.
int fused_cluster_capacity(int S);
int fused_block_capacity();
int fused_cooperative_state();
nvr_status launch_fused_router(const uint16_t* x, float* qrec, float* x_gsa, uint32_t* amax_sync,
                               uint32_t* tile_sync, bool flat, int64_t T, int64_t D,
                               const uint8_t* W_codes, const uint8_t* W_sf, const float* w_gsa, int64_t N,
                               const float* bias, int k, float routed_scaling, bool raw, int32_t* out_ids,
                               float* out_w, float* logits, float* partials, uint32_t* status, int S,
                               int tile_rows, bool test_stall, bool cooperative, cudaStream_t s);
nvr_status launch_router_epilogue(const float* partials, int S, const float* x_gsa, const float* w_gsa,
                                  int64_t T, int64_t N, const float* bias, int k, float routed_scaling,
                                  bool raw, int32_t* out_ids, float* out_w, float* logits, cudaStream_t s);

// ws_words: null, or (for N <= 256) kDecodeWords zeroed words at a fixed
// workspace offset -- then CTA 0 collects the other CTAs' keys by polling
// them (bounded; a timeout goes to *status) instead of the last CTA's ticket.
// test_stall (with ws_words): the other CTAs store no words, so the poll
// runs out.
cudaError_t launch_decode(const void* x, bool bf16, int64_t T, int64_t D, const uint8_t* W_codes,
                          const uint8_t* W_sf, const float* w_gsa, int64_t N, const float* bias,
                          int k, float routed_scaling, bool raw, int32_t* out_ids, float* out_w,
                          float* logits, float* ws_keys, float* ws_scores, uint32_t* ticket,
                          uint64_t* ws_words, uint32_t* status, bool test_stall, const DecodePlan& plan,
                          cudaStream_t s);

}  // namespace nvr
