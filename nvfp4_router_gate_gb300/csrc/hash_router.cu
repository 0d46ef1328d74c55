// hash_router.cu -- router_hash_topk: the token-id router of the first MoE
// layers, one int32 table lookup per (token, slot), no gate GEMM (sm_103a).
//
// Source: "nvfp4-megamoe-kernel commit df05289: dsv4/layers/grouped_linear.py",
// hash-router item (tid2eid is an int32 lookup; nothing to accelerate with a
// GEMM).  With no gate scores, the router's renormalise-and-scale steps see k
// equal scores: every selected expert weighs routed_scaling / k.
//
// One thread per output slot (t, j): consecutive threads write consecutive
// slots, so the id and weight stores are coalesced; the k threads of a token
// read its id once from L1 and its table row (k consecutive int32) in one
// sector or two.  Indices out of range never reach memory: a token id outside
// the table gives -1 / 0 for its row, an entry outside [0, n_experts) -1 / 0
// for its slot.
#include "nvr_internal.h"

namespace nvr {

namespace {

__global__ void __launch_bounds__(256)
hash_router_kernel(const int32_t* __restrict__ token_ids, int64_t n_slots, const int32_t* __restrict__ tid2eid,
                   int64_t vocab, int64_t n_experts, int k, float w_each, int32_t* __restrict__ out_ids,
                   float* __restrict__ out_w) {
  // the token ids may come from the previous kernel of the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_slots; i += stride) {
    const int64_t t = i / k;
    const int j = static_cast<int>(i - t * k);
    const int64_t tid = __ldg(token_ids + t);
    int32_t e = -1;
    if (tid >= 0 && tid < vocab) {
      const int32_t v = __ldg(tid2eid + tid * k + j);
      if (v >= 0 && v < n_experts) e = v;
    }
    out_ids[i] = e;
    out_w[i] = e >= 0 ? w_each : 0.0f;
  }
}

}  // namespace

}  // namespace nvr

extern "C" nvr_status router_hash_topk(const int32_t* token_ids, int64_t T, const int32_t* tid2eid,
                                       int64_t vocab, int64_t n_experts, int k, float routed_scaling,
                                       int32_t* out_ids, float* out_w, nvr_stream_t stream) {
  using namespace nvr;
  if (T < 0 || vocab < 1 || n_experts < 1 || k < 1 || k > kMaxKmax || k > n_experts) return NVR_ERR_INVALID_ARG;
  if (!tid2eid || (T > 0 && (!token_ids || !out_ids || !out_w))) return NVR_ERR_INVALID_ARG;
  if (vocab > (int64_t(1) << 40) || T > (int64_t(1) << 40)) return NVR_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(token_ids) | reinterpret_cast<uintptr_t>(tid2eid) |
       reinterpret_cast<uintptr_t>(out_ids) | reinterpret_cast<uintptr_t>(out_w)) & 3u)
    return NVR_ERR_ALIGNMENT;
  if (T == 0) return NVR_OK;
  const int sms = device_sm_count();
  if (sms <= 0) return NVR_ERR_CUDA;
  const int64_t n_slots = T * k;
  int64_t grid = (n_slots + 255) / 256;
  if (grid > static_cast<int64_t>(sms) * 8) grid = static_cast<int64_t>(sms) * 8;
  // one IEEE division, the same rounding as the scalar definition
  const float w_each = routed_scaling / static_cast<float>(k);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(256);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, hash_router_kernel, token_ids, n_slots, tid2eid, vocab, n_experts,
                                        k, w_each, out_ids, out_w));
}
