// abi.cu -- the extern "C" entry points of include/nvfp4_router.h: argument
// checks (all on the host, before any launch), the workspace layout, and the
// choice between the single-launch decode kernel and the amax -> quantize ->
// tensor-core GEMM+top-k pipeline.
#include <mutex>

#include "nvr_internal.h"

namespace nvr {

TensorMapEncodeFn tensor_map_encoder() {
  static TensorMapEncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<TensorMapEncodeFn>(p);
  });
  return fn;
}

int device_sm_count() {
  static int cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (cache[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = v;
  }
  return cache[dev];
}

int amax_grid(int64_t n_elems, bool bf16, int num_sms) {
  const int64_t nvec = n_elems * (bf16 ? 2 : 4) / 16;
  int64_t want = (nvec + kAmaxThreads * 8 - 1) / (kAmaxThreads * 8);   // >= 8 vectors per thread
  int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 4;
  if (cap > kMaxAmaxGrid) cap = kMaxAmaxGrid;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return static_cast<int>(want);
}

static size_t a256(size_t v) { return (v + 255) / 256 * 256; }

WsLayout quantize_ws_layout(int64_t rows, int64_t D) {
  (void)rows; (void)D;
  WsLayout L;
  L.control = 0;
  L.amax_partials = 256;
  L.scalars = a256(L.amax_partials + kMaxAmaxGrid * 4);
  L.total = L.scalars + 256;
  return L;
}

static int split_bound(int m_tiles, int n_tiles) {
  // the most splits plan_gemm can choose on any GPU with <= 256 SMs
  int s = 256 / (m_tiles > 0 ? m_tiles : 1);
  if (s < 1) s = 1;
  if (s > n_tiles) s = n_tiles;
  if (s > kMaxSplits) s = kMaxSplits;
  return s;
}

WsLayout router_ws_layout(int64_t T, int64_t D, int64_t N) {
  WsLayout L = quantize_ws_layout(T, D);
  const int64_t rows_pad = (T + 127) / 128 * 128;
  const int m_tiles = static_cast<int>(rows_pad / 128);
  const int n_tiles = static_cast<int>((N + 127) / 128);
  // The counters sit at offsets and sizes that do not depend on T: calls of
  // any size may share a workspace sized for the largest, and no call's data
  // regions may cover the words another call expects at zero.
  L.tickets = L.total;
  L.tile_sync = a256(L.tickets + static_cast<size_t>(kMaxTicketTiles) * 4);
  L.dec_words = a256(L.tile_sync + static_cast<size_t>(kMaxFlatTiles) * 8);
  L.x_codes = a256(L.dec_words + static_cast<size_t>(kDecodeWords) * 8);
  L.x_sf = a256(L.x_codes + static_cast<size_t>(rows_pad) * (D / 2));
  L.partials = a256(L.x_sf + static_cast<size_t>(rows_pad) * (D / 16));
  const int splits = split_bound(m_tiles, n_tiles);
  size_t part = splits > 1 ? static_cast<size_t>(m_tiles) * splits * 128 * kMaxKmax * 16 : 0;
  if (N <= 384) {
    // K-split partial logits, rows of 256 (or, for 257-384 experts, 384) floats
    const size_t pk = splitk_partial_rows(T) * (N > 256 ? 384 : 256) * 4;
    if (pk > part) part = pk;
  }
  L.decode = a256(L.partials + part);
  const size_t dec = T <= 16 ? static_cast<size_t>(T) * N * 8 : 0;
  L.total = a256(L.decode + dec);
  return L;
}

}  // namespace nvr

namespace nvr {

thread_local cudaError_t g_last_cuda_error = cudaSuccess;
// nvr_last_router_plan: {kernel sequence, tile rows, CTAs per tile, clustered}
thread_local int g_last_plan[4] = {0, 0, 0, 0};

static void record_plan(int seq, int rows, int per_tile, bool clustered) {
  g_last_plan[0] = seq;
  g_last_plan[1] = rows;
  g_last_plan[2] = per_tile;
  g_last_plan[3] = clustered ? 1 : 0;
}

nvr_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return NVR_OK;
  g_last_cuda_error = e;
  return NVR_ERR_CUDA;
}

// Test hook kernel: holds its SM's shared memory for a bounded time
// (%globaltimer deadline, and an iteration cap), then returns by itself.
__global__ void occupy_kernel(uint64_t ns) {
  extern __shared__ uint8_t held[];
  const uint64_t t0 = globaltimer_ns();
  const uint32_t cap = static_cast<uint32_t>(ns / 500) + 1000;
  for (uint32_t it = 0; it < cap; ++it) {
    if (globaltimer_ns() - t0 >= ns) break;
    __nanosleep(500);
  }
  if (threadIdx.x == 0) held[0] = 1;
}

}  // namespace nvr

using namespace nvr;

namespace {

// measurement hook (nvr_set_profile_events)
void* const* g_prof_events = nullptr;
int g_prof_pairs = 0;

struct ProfileScope {
  cudaStream_t s;
  int i = 0;
  explicit ProfileScope(cudaStream_t st) : s(st) {}
  void before() {
    if (g_prof_events && i < g_prof_pairs) cudaEventRecord(static_cast<cudaEvent_t>(g_prof_events[2 * i]), s);
  }
  void after() {
    if (g_prof_events && i < g_prof_pairs) cudaEventRecord(static_cast<cudaEvent_t>(g_prof_events[2 * i + 1]), s);
    ++i;
  }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

nvr_status check_common(const void* x, nvr_dtype dt, int64_t T, int64_t D, const void* ws) {
  if (!x || !ws) return NVR_ERR_INVALID_ARG;
  if (T < 0 || D <= 0 || D % 64 != 0 || D > (1 << 24)) return NVR_ERR_INVALID_ARG;
  if (dt != NVR_BF16 && dt != NVR_F32) return NVR_ERR_INVALID_ARG;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return NVR_ERR_ALIGNMENT;
  return NVR_OK;
}

nvr_status quantize_impl(const void* x, nvr_dtype dt, int64_t rows, int64_t D, uint8_t* codes,
                         uint8_t* sf, nvr_sf_layout layout, float* gsa, void* ws, size_t ws_bytes,
                         cudaStream_t s) {
  nvr_status st = check_common(x, dt, rows, D, ws);
  if (st != NVR_OK) return st;
  if (!codes || !sf || !gsa) return NVR_ERR_INVALID_ARG;
  if (layout != NVR_SF_LINEAR && layout != NVR_SF_TILED) return NVR_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(sf) || (reinterpret_cast<uintptr_t>(gsa) & 3u)) return NVR_ERR_ALIGNMENT;
  const WsLayout L = quantize_ws_layout(rows, D);
  if (ws_bytes < L.total) return NVR_ERR_WORKSPACE;
  if ((rows + 127) / 128 * 128 * (D / 32) >= (int64_t(1) << 31)) return NVR_ERR_UNSUPPORTED;   // 32-bit indexing
  if (rows == 0) return NVR_OK;
  const int sms = device_sm_count();
  if (sms <= 0) return NVR_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const bool bf16 = dt == NVR_BF16;
  float* qrec = reinterpret_cast<float*>(w + L.scalars + 16);    // {gsa, 1/gsa, mode, amax}
  ProfileScope prof(s);
  prof.before();
  cudaError_t e = launch_amax_bulk(x, bf16, rows * D, reinterpret_cast<uint32_t*>(w + L.amax_partials),
                                   reinterpret_cast<uint32_t*>(w + kWsAmaxTicket), gsa, qrec,
                                   reinterpret_cast<uint32_t*>(w + kWsStatus), sms, s);
  prof.after();
  if (e != cudaSuccess) return cuda_status(e);
  prof.before();
  e = launch_quantize(x, bf16, rows, D, layout == NVR_SF_TILED, qrec, codes, sf, s);
  prof.after();
  return cuda_status(e);
}

constexpr uint32_t kKernelFlags =
    NVR_FLAG_SPLIT_K_2 | NVR_FLAG_SPLIT_K_4 | NVR_FLAG_SPLIT_K_8 | NVR_FLAG_SPLIT_N | NVR_FLAG_STREAM;

// Checks the router flags and folds a kernel-choice flag into
// FORCE_TENSOR_CORE; NVR_ERR_INVALID_ARG for unknown or conflicting flags.
nvr_status normalize_flags(uint32_t& flags) {
  if (flags & ~static_cast<uint32_t>(NVR_FLAG_RAW_LOGITS | NVR_FLAG_FORCE_TENSOR_CORE | NVR_FLAG_FORCE_DECODE |
                                     kKernelFlags | NVR_FLAG_TEST_STALL | NVR_FLAG_NO_COOPERATIVE))
    return NVR_ERR_INVALID_ARG;
  const uint32_t kernel_flags = flags & kKernelFlags;
  if (kernel_flags & (kernel_flags - 1)) return NVR_ERR_INVALID_ARG;          // at most one
  if (kernel_flags) flags |= NVR_FLAG_FORCE_TENSOR_CORE;
  if ((flags & NVR_FLAG_FORCE_TENSOR_CORE) && (flags & NVR_FLAG_FORCE_DECODE)) return NVR_ERR_INVALID_ARG;
  if ((flags & NVR_FLAG_TEST_STALL) && !(flags & (NVR_FLAG_FORCE_TENSOR_CORE | NVR_FLAG_FORCE_DECODE)))
    return NVR_ERR_INVALID_ARG;
  return NVR_OK;
}

// The launch plan of a router call (the sequence codes of nvr_last_router_plan).
struct RouterPlan {
  int seq = 0;                 // 1 decode, 2 fused, 3 amax + fused, 4 amax + quantize + K split + epilogue,
                               // 5 amax + quantize + N split, 6 amax + quantize + weight streaming
  int tile_rows = 0, per_tile = 0;
  bool clustered = false;      // seq 1: decode clusters; seq 2-3: the tile's CTAs form a cluster
  DecodePlan dp;               // seq 1
  GemmPlan g;                  // seq 5
};

// The plan for T > 0 tokens on a device with `sms` SMs that holds
// cluster_cap[i] clusters of 2^i CTAs of the fused kernel at once (i = 0..4)
// and block_cap of its CTAs without clusters.  Host arithmetic only: the
// dispatch and nvr_plan_router both call it.  flags: normalised.
//
// The fused kernel (bf16, <= 384 experts): token tiles of 128 or 112 rows,
// S CTAs per tile (S a power of two no larger than the K-split plan; each CTA
// routes rows/S tokens) that form a cluster or, without clusters, meet at a
// barrier in the workspace.  Among the grids resident at once the one with
// the least work per CTA (rows x K stages per CTA) wins, clusters on a tie;
// the device holds fewer CTAs in clusters than without (whole clusters per
// GPC), so at T = 4096 112-row tiles put 148 CTAs on the SMs without clusters
// where clusters of 4 hold 128.  Forced split factors keep 128-row tiles.
// With no resident grid: clusters, after the amax kernel.
nvr_status plan_router(int64_t T, int64_t D, int64_t N, bool bf16, uint32_t flags, int sms,
                       const int (&cluster_cap)[5], int block_cap, RouterPlan& rp) {
  const int forced_split = (flags & NVR_FLAG_SPLIT_K_2) ? 2 : (flags & NVR_FLAG_SPLIT_K_4) ? 4
                           : (flags & NVR_FLAG_SPLIT_K_8) ? 8 : 0;
  if (forced_split && N > 256) return NVR_ERR_UNSUPPORTED;
  rp.dp = plan_decode(T, D, N, sms, bf16);
  const bool use_decode = (flags & NVR_FLAG_FORCE_DECODE) ? true
                          : (flags & NVR_FLAG_FORCE_TENSOR_CORE) ? false
                          : rp.dp.ok;
  if (use_decode) {
    if (!rp.dp.ok) return NVR_ERR_UNSUPPORTED;
    rp.seq = 1;
    rp.clustered = rp.dp.cluster > 1;
    return NVR_OK;
  }
  // Up to 256 experts (bf16: 384): K split over S CTAs with one tensor-core
  // accumulator for the whole row each; bf16 activations are quantized inside
  // the GEMM and routed in the same kernel, fp32 ones take the standalone
  // quantizer, the K-split GEMM and the epilogue kernel.  Wider heads, after
  // the standalone quantize kernel: up to 128 tokens stream the weight (its
  // 128-row tiles as the MMA's M, the tokens as its N), more tokens split the
  // N tiles across CTAs; both merge the per-token top-k lists across CTAs.
  const int split_k = forced_split ? forced_split
                      : (flags & (NVR_FLAG_SPLIT_N | NVR_FLAG_STREAM)) || N > (bf16 ? 384 : 256)
                          ? 0
                          : plan_splitk(T, D, sms);
  if (split_k > 0 && bf16) {
    const int n_st = static_cast<int>((D / kBlock + 15) / 16);
    int tile_rows = 128, S = 1;
    bool one_launch = false, flat = false;
    int64_t best = -1;
    for (int rows : {128, 112}) {
      if (forced_split && rows != 128) continue;
      const int64_t m_tiles = (T + rows - 1) / rows;
      for (int c = 16, ci = 4; c >= 1; c >>= 1, --ci) {
        if (forced_split ? c != forced_split : c > split_k) continue;
        const int64_t cost = static_cast<int64_t>(rows) * ((n_st + c - 1) / c);
        for (int f = 0; f < (c > 1 ? 2 : 1); ++f) {
          const bool resident = f ? m_tiles * c <= block_cap && m_tiles <= kMaxFlatTiles
                                  : cluster_cap[ci] >= m_tiles;
          if (f && !resident) continue;
          if (best < 0 || (resident && !one_launch) || (resident == one_launch && cost < best)) {
            best = cost;
            tile_rows = rows;
            S = c;
            flat = f != 0;
            one_launch = resident;
          }
        }
      }
    }
    rp.seq = one_launch ? 2 : 3;
    rp.tile_rows = tile_rows;
    rp.per_tile = S;
    rp.clustered = !flat;
    return NVR_OK;
  }
  if (split_k > 0) {
    rp.seq = 4;
    rp.tile_rows = 128;
    rp.per_tile = split_k;
    return NVR_OK;
  }
  if ((flags & NVR_FLAG_STREAM) || (!(flags & NVR_FLAG_SPLIT_N) && T <= 128)) {
    if (T > 128) return NVR_ERR_UNSUPPORTED;
    rp.seq = 6;
    rp.tile_rows = stream_token_tile(T);
    rp.per_tile = stream_splits(N, sms);
    return NVR_OK;
  }
  rp.g = plan_gemm(T, N, sms);
  if (rp.g.m_tiles > kMaxTicketTiles) return NVR_ERR_UNSUPPORTED;
  rp.seq = 5;
  rp.tile_rows = 128;
  rp.per_tile = rp.g.n_splits;
  return NVR_OK;
}

nvr_status router_impl(const void* x, nvr_dtype dt, int64_t T, int64_t D, const uint8_t* W_fp4,
                       const uint8_t* W_sf, const float* w_gsa, int64_t N, const float* bias, int k,
                       float routed_scaling, uint32_t flags, int32_t* out_ids, float* out_w,
                       void* out_logits, bool logits_bf16, void* ws, size_t ws_bytes, cudaStream_t s) {
  // logits mode (out_logits set): fp32 on every path; bf16 only on the
  // streaming and N-split kernels (the callers force one of them)
  float* logits = static_cast<float*>(out_logits);
  nvr_status st = check_common(x, dt, T, D, ws);
  if (st != NVR_OK) return st;
  if (!W_fp4 || !W_sf || !w_gsa || N <= 0 || N > (1 << 28)) return NVR_ERR_INVALID_ARG;
  if (!logits && (!out_ids || !out_w || k < 1 || k > kMaxKmax || k > N)) return NVR_ERR_INVALID_ARG;
  st = normalize_flags(flags);
  if (st != NVR_OK) return st;
  if ((flags & kKernelFlags & ~static_cast<uint32_t>(NVR_FLAG_SPLIT_N | NVR_FLAG_STREAM)) && N > 256)
    return NVR_ERR_UNSUPPORTED;
  if (!aligned16(W_fp4) || !aligned16(W_sf) || (reinterpret_cast<uintptr_t>(w_gsa) & 3u) ||
      (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)) ||
      (out_ids && (reinterpret_cast<uintptr_t>(out_ids) & 3u)) ||
      (out_w && (reinterpret_cast<uintptr_t>(out_w) & 3u)) ||
      (logits && (reinterpret_cast<uintptr_t>(logits) & 3u)))
    return NVR_ERR_ALIGNMENT;
  const WsLayout L = router_ws_layout(T, D, N);
  if (ws_bytes < L.total) return NVR_ERR_WORKSPACE;
  if ((T + 127) / 128 * 128 * (D / 32) >= (int64_t(1) << 31)) return NVR_ERR_UNSUPPORTED;      // 32-bit indexing
  if (T == 0) return NVR_OK;
  const int sms = device_sm_count();
  if (sms <= 0) return NVR_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const bool bf16 = dt == NVR_BF16;
  const bool raw = (flags & NVR_FLAG_RAW_LOGITS) != 0;
  if (logits) k = 1;

  // the fused kernel's capacities, queried (once per device) only where it
  // may run -- never for a decode call, which may be the first call of a
  // process and inside a graph capture
  const bool maybe_fused = bf16 && N <= 384 &&
                           !(flags & (NVR_FLAG_SPLIT_N | NVR_FLAG_STREAM | NVR_FLAG_FORCE_DECODE)) &&
                           ((flags & NVR_FLAG_FORCE_TENSOR_CORE) || !plan_decode(T, D, N, sms, bf16).ok);
  int cluster_cap[5] = {0, 0, 0, 0, 0};
  int block_cap = 0;
  if (maybe_fused) {
    for (int i = 0; i < 5; ++i) cluster_cap[i] = fused_cluster_capacity(1 << i);
    block_cap = fused_block_capacity();
  }
  RouterPlan rp;
  st = plan_router(T, D, N, bf16, flags, sms, cluster_cap, block_cap, rp);
  if (st != NVR_OK) return st;
  if (logits_bf16 && rp.seq != 5 && rp.seq != 6) return NVR_ERR_UNSUPPORTED;
  record_plan(rp.seq, rp.tile_rows, rp.per_tile, rp.clustered);
  if (rp.seq == 1) {
    float* keys = reinterpret_cast<float*>(w + L.decode);
    float* scores = keys + T * N;
    ProfileScope prof(s);
    prof.before();
    // up to 256 experts CTA 0 collects the keys from the fixed words region
    uint64_t* words = N <= 256 ? reinterpret_cast<uint64_t*>(w + L.dec_words) : nullptr;
    cudaError_t e = launch_decode(x, bf16, T, D, W_fp4, W_sf, w_gsa, N, bias, k, routed_scaling, raw,
                                  out_ids, out_w, logits, keys, scores,
                                  reinterpret_cast<uint32_t*>(w + kWsDecodeTicket), words,
                                  reinterpret_cast<uint32_t*>(w + kWsStatus),
                                  (flags & NVR_FLAG_TEST_STALL) != 0, rp.dp, s);
    prof.after();
    return cuda_status(e);
  }
  float* x_gsa = reinterpret_cast<float*>(w + L.scalars);
  float* qrec = x_gsa + 4;                                        // {gsa, 1/gsa, mode, amax}
  uint8_t* xc = w + L.x_codes;
  uint8_t* xsf = w + L.x_sf;
  uint32_t* status = reinterpret_cast<uint32_t*>(w + kWsStatus);
  const bool stall = (flags & NVR_FLAG_TEST_STALL) != 0;
  ProfileScope prof(s);
  float* partials = reinterpret_cast<float*>(w + L.partials);
  if (rp.seq == 2 || rp.seq == 3) {
    const bool one_launch = rp.seq == 2, flat = !rp.clustered;
    if (!one_launch) {
      prof.before();
      const cudaError_t e = launch_amax_bulk(x, bf16, T * D, reinterpret_cast<uint32_t*>(w + L.amax_partials),
                                             reinterpret_cast<uint32_t*>(w + kWsAmaxTicket), x_gsa, qrec, status,
                                             sms, s);
      prof.after();
      if (e != cudaSuccess) return cuda_status(e);
    }
    prof.before();
    st = launch_fused_router(static_cast<const uint16_t*>(x), qrec, x_gsa,
                             one_launch ? reinterpret_cast<uint32_t*>(w + kWsFusedAmax) : nullptr,
                             one_launch ? reinterpret_cast<uint32_t*>(w + L.tile_sync) : nullptr, flat, T, D, W_fp4,
                             W_sf, w_gsa, N, bias, k, routed_scaling, raw, out_ids, out_w, logits, partials, status,
                             rp.per_tile, rp.tile_rows, stall, (flags & NVR_FLAG_NO_COOPERATIVE) == 0, s);
    prof.after();
    return st;
  }
  const int split_k = rp.seq == 4 ? rp.per_tile : 0;
  prof.before();
  cudaError_t e = launch_amax_bulk(x, bf16, T * D, reinterpret_cast<uint32_t*>(w + L.amax_partials),
                                   reinterpret_cast<uint32_t*>(w + kWsAmaxTicket), x_gsa, qrec, status, sms, s);
  prof.after();
  if (e != cudaSuccess) return cuda_status(e);
  prof.before();
  e = launch_quantize(x, bf16, T, D, true, qrec, xc, xsf, s);
  prof.after();
  if (e != cudaSuccess) return cuda_status(e);
  if (rp.seq == 6) {
    prof.before();
    st = launch_gemm_stream(xc, xsf, x_gsa, T, D, W_fp4, W_sf, w_gsa, N, bias, k, routed_scaling, raw, out_ids,
                            out_w, out_logits, logits_bf16, reinterpret_cast<float4*>(w + L.partials),
                            reinterpret_cast<uint32_t*>(w + L.tickets), status, rp.per_tile, stall, s);
    prof.after();
    return st;
  }
  if (split_k > 0) {
    prof.before();
    st = launch_splitk_gemm(xc, xsf, T, D, W_fp4, W_sf, N, partials, status, split_k, stall, s);
    prof.after();
    if (st != NVR_OK) return st;
    prof.before();
    st = launch_router_epilogue(partials, split_k, x_gsa, w_gsa, T, N, bias, k, routed_scaling, raw, out_ids,
                                out_w, logits, s);
    prof.after();
    return st;
  }
  prof.before();
  st = launch_gemm_topk(xc, xsf, x_gsa, T, D, W_fp4, W_sf, w_gsa, N, bias, k, routed_scaling, raw,
                        out_ids, out_w, out_logits, logits_bf16, reinterpret_cast<float4*>(w + L.partials),
                        reinterpret_cast<uint32_t*>(w + L.tickets), status, rp.g, stall, s);
  prof.after();
  return st;
}

}  // namespace

extern "C" {

const char* nvr_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda_error); }

nvr_status nvr_plan_router(int64_t T, int64_t D, int64_t N, nvr_dtype dt, uint32_t flags, int num_sms,
                           const int* cluster_capacity, int block_capacity, int* out) {
  if (!cluster_capacity || !out) return NVR_ERR_INVALID_ARG;
  if (T < 1 || D <= 0 || D % 64 != 0 || D > (1 << 24) || N <= 0 || N > (1 << 28)) return NVR_ERR_INVALID_ARG;
  if (dt != NVR_BF16 && dt != NVR_F32) return NVR_ERR_INVALID_ARG;
  if (num_sms < 1 || block_capacity < 0) return NVR_ERR_INVALID_ARG;
  nvr_status st = normalize_flags(flags);
  if (st != NVR_OK) return st;
  int caps[5];
  for (int i = 0; i < 5; ++i) caps[i] = cluster_capacity[i];
  RouterPlan rp;
  st = plan_router(T, D, N, dt == NVR_BF16, flags, num_sms, caps, block_capacity, rp);
  if (st != NVR_OK) return st;
  out[0] = rp.seq;
  out[1] = rp.tile_rows;
  out[2] = rp.per_tile;
  out[3] = rp.clustered ? 1 : 0;
  return NVR_OK;
}

int nvr_router_cooperative_state(void) { return fused_cooperative_state(); }

nvr_status nvr_test_occupy(int n_ctas, int smem_bytes, uint64_t duration_ns, nvr_stream_t stream) {
  if (n_ctas < 1 || n_ctas > 65536 || smem_bytes < 0 || smem_bytes > 227 * 1024 || duration_ns > 1000000000ull)
    return NVR_ERR_INVALID_ARG;
  cudaError_t e = cudaFuncSetAttribute(occupy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return cuda_status(e);
  occupy_kernel<<<n_ctas, 32, smem_bytes, reinterpret_cast<cudaStream_t>(stream)>>>(duration_ns);
  return cuda_status(cudaGetLastError());
}

nvr_status nvr_last_router_plan(int* out) {
  if (!out) return NVR_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i) out[i] = g_last_plan[i];
  return NVR_OK;
}

const char* nvr_status_string(nvr_status s) {
  switch (s) {
    case NVR_OK: return "ok";
    case NVR_ERR_INVALID_ARG: return "invalid argument";
    case NVR_ERR_UNSUPPORTED: return "unsupported shape or configuration";
    case NVR_ERR_ALIGNMENT: return "pointer not aligned (16 bytes for arrays, 256 for the workspace)";
    case NVR_ERR_WORKSPACE: return "workspace too small";
    case NVR_ERR_CUDA: return "CUDA error";
    case NVR_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

size_t nvr_sf_bytes(int64_t rows, int64_t D, nvr_sf_layout layout) {
  if (rows < 0 || D <= 0 || D % 64 != 0) return 0;
  if (layout == NVR_SF_LINEAR) return static_cast<size_t>(rows) * (D / 16);
  if (layout == NVR_SF_TILED) return static_cast<size_t>((rows + 127) / 128 * 128) * (D / 16);
  return 0;
}

size_t nvfp4_quantize_workspace_size(int64_t rows, int64_t D) {
  return quantize_ws_layout(rows, D).total;
}

nvr_status nvfp4_quantize_act(const void* x, nvr_dtype dt, int64_t T, int64_t D, uint8_t* x_fp4,
                              uint8_t* x_sf, nvr_sf_layout sf_layout, float* x_gsa, void* workspace,
                              size_t ws_bytes, nvr_stream_t stream) {
  return quantize_impl(x, dt, T, D, x_fp4, x_sf, sf_layout, x_gsa, workspace, ws_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

nvr_status nvfp4_pack_weight(const void* W, nvr_dtype dt, int64_t N, int64_t D, uint8_t* W_fp4,
                             uint8_t* W_sf, float* w_gsa, void* workspace, size_t ws_bytes,
                             nvr_stream_t stream) {
  return quantize_impl(W, dt, N, D, W_fp4, W_sf, NVR_SF_TILED, w_gsa, workspace, ws_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

size_t router_gate_workspace_size(int64_t T_max, int64_t D, int64_t N, int k) {
  (void)k;
  if (T_max < 0 || D <= 0 || D % 64 != 0 || N <= 0) return 0;
  // An upper bound of router_ws_layout(T, D, N).total over every T <= T_max:
  // the split-partials and decode regions do not grow monotonically with T.
  const int64_t rows_pad = (T_max + 127) / 128 * 128;
  const int m_max = static_cast<int>(rows_pad / 128);
  const int n_tiles = static_cast<int>((N + 127) / 128);
  size_t part = 0;
  for (int m = 1; m <= m_max; ++m) {
    const int sp = split_bound(m, n_tiles);
    if (sp > 1) {
      const size_t v = static_cast<size_t>(m) * sp * 128 * kMaxKmax * 16;
      if (v > part) part = v;
    }
  }
  if (N <= 384) {
    const size_t pk = splitk_partial_rows(T_max) * (N > 256 ? 384 : 256) * 4;   // monotone in T
    if (pk > part) part = pk;
  }
  const int64_t t_dec = T_max < 16 ? T_max : 16;
  return quantize_ws_layout(T_max, D).total + static_cast<size_t>(kMaxTicketTiles) * 4 +
         static_cast<size_t>(kMaxFlatTiles) * 8 + static_cast<size_t>(kDecodeWords) * 8 +
         static_cast<size_t>(rows_pad) * (D / 2) + static_cast<size_t>(rows_pad) * (D / 16) + part +
         static_cast<size_t>(t_dec) * N * 8 + 9 * 256;
}

size_t router_gate_x_gsa_offset(void) { return router_ws_layout(1, 64, 1).scalars; }

nvr_status router_gate_topk(const void* x, nvr_dtype dt, int64_t T, int64_t D, const uint8_t* W_fp4,
                            const uint8_t* W_scales, const float* w_gsa, int64_t N, const float* bias,
                            int k, float routed_scaling, uint32_t flags, int32_t* out_ids,
                            float* out_w, void* workspace, size_t ws_bytes, nvr_stream_t stream) {
  if (!out_ids || !out_w) return NVR_ERR_INVALID_ARG;
  return router_impl(x, dt, T, D, W_fp4, W_scales, w_gsa, N, bias, k, routed_scaling, flags, out_ids,
                     out_w, nullptr, false, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

nvr_status router_gate_logits(const void* x, nvr_dtype dt, int64_t T, int64_t D, const uint8_t* W_fp4,
                              const uint8_t* W_scales, const float* w_gsa, int64_t N, uint32_t flags,
                              float* logits, void* workspace, size_t ws_bytes, nvr_stream_t stream) {
  if (!logits) return NVR_ERR_INVALID_ARG;
  if (flags & (NVR_FLAG_RAW_LOGITS | NVR_FLAG_TEST_STALL)) return NVR_ERR_INVALID_ARG;
  return router_impl(x, dt, T, D, W_fp4, W_scales, w_gsa, N, nullptr, 1, 1.0f, flags, nullptr, nullptr,
                     logits, false, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t nvfp4_linear_workspace_size(int64_t T_max, int64_t D, int64_t N) {
  return router_gate_workspace_size(T_max, D, N, 1);
}

nvr_status nvfp4_linear(const void* x, nvr_dtype dt, int64_t T, int64_t D, const uint8_t* W_fp4,
                        const uint8_t* W_scales, const float* w_gsa, int64_t N, void* out, nvr_dtype out_dt,
                        void* workspace, size_t ws_bytes, nvr_stream_t stream) {
  if (!out) return NVR_ERR_INVALID_ARG;
  if (out_dt != NVR_BF16 && out_dt != NVR_F32) return NVR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(out) & 15u) return NVR_ERR_ALIGNMENT;
  // up to 128 tokens stream the weight; more take the token-tiled N-split GEMM
  const uint32_t flags = T <= 128 ? NVR_FLAG_STREAM : NVR_FLAG_SPLIT_N;
  return router_impl(x, dt, T, D, W_fp4, W_scales, w_gsa, N, nullptr, 1, 1.0f, flags, nullptr, nullptr, out,
                     out_dt == NVR_BF16, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

nvr_status nvr_set_profile_events(void* const* events, int n_pairs) {
  if (events && n_pairs > 0) {
    g_prof_events = events;
    g_prof_pairs = n_pairs;
  } else {
    g_prof_events = nullptr;
    g_prof_pairs = 0;
  }
  return NVR_OK;
}

nvr_status nvr_read_device_status(const void* workspace, nvr_stream_t stream, nvr_status* out) {
  if (!workspace || !out) return NVR_ERR_INVALID_ARG;
  uint32_t v = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, static_cast<const uint8_t*>(workspace) + kWsStatus, 4, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return NVR_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return NVR_ERR_CUDA;
  *out = static_cast<nvr_status>(v);
  return NVR_OK;
}

}  // extern "C"
