/*
 * nvfp4_router.h -- C ABI of the GB300 (sm_103a) NVFP4 MoE router gate.
 *
 * One router call turns a batch of token activations x [T, D] into, per token,
 * the k selected expert ids and their routing weights:
 *
 *   1. runtime NVFP4 quantization of x: one global scale per call,
 *      gsa = max|x| / (6 * 448), 16-element blocks along D with an E4M3 scale
 *      byte each and E2M1 4-bit codes
 *      ("nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py",
 *      runtime-gsa section; "commit df05289: dsv4/layers/grouped_linear.py",
 *      zero-sync fused quantize section);
 *   2. the block-scaled NVFP4 gate GEMM  logits = x . W_gate^T  against
 *      NVFP4-packed expert weights (router.py page, NVFP4 gate section);
 *   3. the fused "activation_topk" epilogue: sigmoid scores, top-k on
 *      score + bias, gather of the unbiased scores, renormalisation by their
 *      sum and multiplication by routed_scaling, written as int32 ids and fp32
 *      weights ("commit e0f60b9: dsv4/kernels/router/__init__.py",
 *      activation_topk section).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All array pointers are DEVICE pointers owned by the caller.  The library
 *   never allocates or frees device memory and keeps no per-call host state;
 *   the only global state is a per-device cache of attributes (SM count,
 *   kernel attributes), set on first use.
 * - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t,
 *   NULL = legacy default stream).  They never synchronise the host and never
 *   copy the global scales to the host, so they can be captured in a CUDA
 *   graph.  Errors found on the host are returned before any launch.
 * - Arguments checked on the host (status NVR_ERR_INVALID_ARG unless noted):
 *   null pointers; T < 0, D <= 0, D % 64 != 0, N <= 0; dtype not BF16/F32;
 *   k < 1, k > 16, k > N; array pointers not 16-byte aligned
 *   (NVR_ERR_ALIGNMENT); workspace smaller than the size query returns
 *   (NVR_ERR_WORKSPACE).  T == 0 is a valid empty call that launches nothing.
 * - A failed launch returns NVR_ERR_CUDA (the CUDA error is consumed).
 * - Device-side bounded waits that time out (never expected in a correct
 *   build; each wait is limited to about one second) store NVR_ERR_TIMEOUT in
 *   the workspace status word, which nvr_read_device_status returns.
 * - Workspace: caller-allocated device memory of at least the size the
 *   matching *_workspace_size function returns, 256-byte aligned, ZEROED ONCE
 *   before first use.  Every call leaves its counters ready for the next, so the
 *   same workspace serves any number of calls on one stream, of any T up to
 *   the T_max it was sized for (the counters sit at fixed offsets, outside the
 *   regions whose size depends on T).  Calls that share
 *   a workspace must not run concurrently.  After a call that returned an
 *   error or timed out, zero the workspace again.
 * - Non-finite inputs (NaN, Inf) are outside the contract: the output is
 *   unspecified but the kernels do not fault.
 *
 * Data layouts
 * ------------
 * - x: [T, D] row-major, bf16 (NVR_BF16) or fp32 (NVR_F32).
 * - packed codes: [rows, D/2] uint8, element 2j in the low nibble of byte j.
 * - scale bytes, NVR_SF_LINEAR: [rows, D/16] uint8 row-major.
 * - scale bytes, NVR_SF_TILED: the tensor-core tile layout: tiles of 128 rows
 *   x 4 scale columns (512 bytes); inside a tile the byte of (row r, column c)
 *   sits at 16*(r%32) + 4*((r%128)/32) + (c%4); tile (r/128, c/4) starts at
 *   ((r/128)*(D/64) + c/4) * 512.  Rows are padded to a multiple of 128 with
 *   zero bytes; the buffer holds nvr_sf_bytes(rows, D, NVR_SF_TILED) bytes.
 * - global scales: one fp32 in device memory.
 */
#ifndef NVFP4_ROUTER_H
#define NVFP4_ROUTER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* nvr_stream_t; /* the same handle as cudaStream_t */

typedef enum {
  NVR_OK = 0,
  NVR_ERR_INVALID_ARG = 1,
  NVR_ERR_UNSUPPORTED = 2,
  NVR_ERR_ALIGNMENT = 3,
  NVR_ERR_WORKSPACE = 4,
  NVR_ERR_CUDA = 5,
  NVR_ERR_TIMEOUT = 6
} nvr_status;

typedef enum { NVR_BF16 = 0, NVR_F32 = 1 } nvr_dtype;

typedef enum { NVR_SF_LINEAR = 0, NVR_SF_TILED = 1 } nvr_sf_layout;

/* router_gate_topk flags */
enum {
  /* Raw-logit head: no sigmoid, bias, renormalisation or scaling.  The top-k
   * is taken on the fp32 logits and out_w receives the selected logits. */
  NVR_FLAG_RAW_LOGITS = 1u,
  /* Kernel choice for tests and benchmarks.  By default the shape decides:
   * T <= 16 tokens (with T*D and N small enough for one CTA's shared memory)
   * run the single-launch decode kernel, everything else the tensor-core
   * pipeline.  FORCE_TENSOR_CORE always takes the tensor-core pipeline;
   * FORCE_DECODE takes the single-launch kernel or returns
   * NVR_ERR_UNSUPPORTED when the shape is outside its limits.  Both give
   * results within the same tolerances; they are not bit-identical (the
   * fp32 accumulation order of the logits differs). */
  NVR_FLAG_FORCE_TENSOR_CORE = 2u,
  NVR_FLAG_FORCE_DECODE = 4u,
  /* Tensor-core kernel choice (each implies FORCE_TENSOR_CORE; at most one).
   * By default heads of up to 256 experts (bf16 x: 384) split K over a
   * cluster of S CTAs
   * per token tile (S and the tile height, 128 or 112 rows, from T, D and
   * the number of clusters the device holds at once; fp32 partial logits
   * pass through the workspace, L2-resident, to the CTAs of the same
   * cluster, which route the tile's tokens), and wider heads split N across
   * CTAs.  SPLIT_K_2/4/8 force S with 128-row tiles (NVR_ERR_UNSUPPORTED
   * when N > 256); SPLIT_N forces the N-split kernel for any N.  Results
   * agree within the same tolerances; the logits' fp32 summation order
   * differs. */
  NVR_FLAG_SPLIT_K_2 = 8u,
  NVR_FLAG_SPLIT_K_4 = 16u,
  NVR_FLAG_SPLIT_K_8 = 32u,
  NVR_FLAG_SPLIT_N = 64u,
  /* Forces the weight-streaming kernel (T <= 128; NVR_ERR_UNSUPPORTED for
   * more tokens): the 128-row weight tiles are the MMA's M and the tokens its
   * N, the weight is read once, per-token top-k lists are merged across CTAs.
   * The default for heads of more than 384 experts (fp32 x: 256) at
   * T <= 128. */
  NVR_FLAG_STREAM = 128u,
  /* The one-launch prefill router is launched cooperatively by default (the
   * runtime then guarantees that its whole grid is resident at once, which
   * its grid barrier needs even while other streams' kernels hold SMs; see
   * nvr_router_cooperative_state).  A cooperative grid cannot start while the
   * previous kernel of the stream is still draining, which costs about 3 us
   * per call back to back on a GB300.  This flag launches it as an ordinary
   * programmatic dependent launch instead: for callers that know no other
   * work holds the SMs during the call (the host's occupancy check and the
   * barriers' bounded waits are then the only safeguards; a wait that runs
   * out records NVR_ERR_TIMEOUT in the workspace). */
  NVR_FLAG_NO_COOPERATIVE = 256u,
  /* Failure-detection test hook (with FORCE_TENSOR_CORE or a SPLIT flag): the tensor-core
   * kernel's MMA issuer issues nothing, so its bounded waits run out after
   * about one second; the kernel stores NVR_ERR_TIMEOUT in the workspace
   * status word, releases its tensor memory and returns.  With FORCE_DECODE
   * (up to 256 experts): the decode CTAs other than the collector store no
   * keys, so the collector's poll runs out after about one second and stores
   * NVR_ERR_TIMEOUT.  The call itself returns NVR_OK (the failure is on the
   * device); outputs are unspecified. */
  NVR_FLAG_TEST_STALL = 1u << 30
};

/* Human-readable name of a status code (static string, never NULL). */
const char* nvr_status_string(nvr_status s);

/* Name of the CUDA error behind the most recent NVR_ERR_CUDA returned to this
 * host thread ("cudaSuccess" if none; static string, never NULL).  No
 * counterpart on the pages: a diagnostic for launch failures. */
const char* nvr_last_cuda_error(void);

/* The launch plan of the most recent router_gate_topk / router_gate_logits
 * call that reached a launch on this host thread, as four ints:
 *   out[0] kernel sequence: 0 none yet, 1 the decode kernel, 2 the one-launch
 *          fused router, 3 amax then the fused router, 4 amax, quantize,
 *          K-split GEMM and epilogue kernel, 5 amax, quantize and the
 *          N-split GEMM, 6 amax, quantize and the weight-streaming GEMM;
 *   out[1] token-tile rows (128 or 112; for sequence 6 the token columns of
 *          the MMA, 32, 64 or 128; 0 for sequences 0, 1);
 *   out[2] CTAs per token tile (K splits for 2-4, N splits for 5 and 6; 0 for
 *          0, 1);
 *   out[3] 1 when the CTAs of a tile form a thread-block cluster, else 0.
 * No counterpart on the pages: a diagnostic for tests and benchmarks.
 * NVR_ERR_INVALID_ARG for a NULL out. */
nvr_status nvr_last_router_plan(int* out);

/* Whether the one-launch prefill router (plan sequence 2) is launched
 * cooperatively on the current device: 1 yes (the runtime guarantees that its
 * whole grid is resident at once, which its grid barrier needs, also next to
 * other kernels), -1 the runtime refused the cooperative attribute together
 * with programmatic launch and clusters (the host's occupancy check and the
 * barriers' bounded waits remain), 0 not known yet (found out on the first
 * one-launch call outside stream capture).  No counterpart on the pages. */
int nvr_router_cooperative_state(void);

/* nvr_test_occupy -- test hook (no counterpart on the pages): launches n_ctas
 * CTAs on `stream` that each hold smem_bytes of shared memory (at most 227 KB)
 * and return by themselves after duration_ns (at most one second; a
 * %globaltimer deadline and an iteration cap), so that a test can run router
 * calls while other work holds the SMs.  NVR_ERR_INVALID_ARG outside those
 * bounds. */
nvr_status nvr_test_occupy(int n_ctas, int smem_bytes, uint64_t duration_ns, nvr_stream_t stream);

/* nvr_test_conversion_sweep -- test hook: checks the hardware conversions
 * behind every quantizer path, cvt.rn.satfinite.e2m1x2.f32 (E2M1 codes) and
 * cvt.rn.satfinite.e4m3x2.f32 (E4M3 scale bytes), on every float32 bit pattern
 * except the NaNs, in both halves of each paired conversion.  The formats are
 * the standard E2M1 and E4M3 ("fn") with the maxima the pages fix (6 and 448;
 * "nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py", runtime-gsa
 * section), rounding to nearest, ties to the even code, saturating.
 *   th_e2m1  device, 7 uint32: t_1..t_7, t_i the smallest float32 bit pattern
 *            whose E2M1 magnitude code is >= i (ascending);
 *   th_e4m3  device, 126 uint32: the same for the E4M3 magnitude codes
 *            0x01..0x7E;
 *   counts   device, 3 uint64 (written): E2M1 mismatches, E4M3 mismatches,
 *            inputs checked (2^32 - 2^24 + 2);
 *   first    device, 2 uint32 (written): the smallest mismatching bit
 *            pattern of each conversion, 0xFFFFFFFF if none.
 * A conversion matches when its magnitude code is #{i : bits(|x|) >= t_i}
 * and, for a nonzero code, its sign bit is the input's (the sign of a zero
 * result is not compared).  Asynchronous on `stream` (it zeroes counts and
 * first first); NVR_ERR_INVALID_ARG for a null pointer.  A few ms. */
nvr_status nvr_test_conversion_sweep(const uint32_t* th_e2m1, const uint32_t* th_e4m3,
                                     unsigned long long* counts, uint32_t* first, nvr_stream_t stream);

/* nvr_plan_router -- the launch plan router_gate_topk would choose for a call
 * of T >= 1 tokens (dtype dt, hidden D, N experts, flags as for
 * router_gate_topk) on a device with num_sms SMs that holds
 * cluster_capacity[i] clusters of 2^i CTAs of the fused router kernel at once
 * (i = 0..4, five ints) and block_capacity of its CTAs without clusters.  Host
 * arithmetic only (no device access): the dispatch runs the same function
 * with the current device's capacities.  out: the four ints described at
 * nvr_last_router_plan.  NVR_ERR_INVALID_ARG for NULL pointers, a shape or
 * flags router_gate_topk would reject, num_sms < 1; NVR_ERR_UNSUPPORTED where
 * router_gate_topk would return it for the shape (a forced decode that does
 * not fit, a forced K split with N > 256).  No counterpart on the pages: a
 * diagnostic for capacity planning and tests. */
nvr_status nvr_plan_router(int64_t T, int64_t D, int64_t N, nvr_dtype dt, uint32_t flags, int num_sms,
                           const int* cluster_capacity, int block_capacity, int* out);

/* Bytes of a scale-byte buffer for [rows, D] in the given layout
 * (0 for invalid arguments). */
size_t nvr_sf_bytes(int64_t rows, int64_t D, nvr_sf_layout layout);

/* Workspace bytes nvfp4_quantize_act / nvfp4_pack_weight need for up to
 * `rows` rows of length D. */
size_t nvfp4_quantize_workspace_size(int64_t rows, int64_t D);

/*
 * nvfp4_quantize_act -- runtime NVFP4 quantization of one activation tensor.
 *
 * Source: "nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py",
 * runtime-gsa section (gsa = max|x| / (6.0 * 448.0), so x/gsa <= 2688), and
 * "commit df05289: dsv4/layers/grouped_linear.py", zero-sync fused quantize
 * section (all rows flattened into one tensor, one global scale, computed
 * and kept on the GPU).
 *
 * Computes, in IEEE fp32 with round-to-nearest-even:
 *   amax = max |x| over all T*D elements; *x_gsa = amax / 2688;
 *   per element y = x / gsa; per 16-element block sy = max|y| / 6,
 *   scale byte = E4M3(sy) (nearest-even, saturating at 448);
 *   code = E2M1(y / dec(byte)) (nearest-even, saturating at 6, sign kept);
 *   a block whose scale byte is 0 has all codes 0; amax == 0 gives gsa 0 and
 *   all-zero output.
 *
 *   x         [T, D] input (bf16 or fp32 per dt), 16-byte aligned
 *   x_fp4     out [T, D/2] packed codes
 *   x_sf      out scale bytes in `sf_layout` (nvr_sf_bytes(T, D, sf_layout))
 *   x_gsa     out, one fp32 (device)
 *   workspace nvfp4_quantize_workspace_size(T, D) bytes, zeroed once
 * Two kernels (amax with a grid-level reduce, then quantize); no host sync.
 */
nvr_status nvfp4_quantize_act(const void* x, nvr_dtype dt, int64_t T, int64_t D,
                              uint8_t* x_fp4, uint8_t* x_sf, nvr_sf_layout sf_layout,
                              float* x_gsa, void* workspace, size_t ws_bytes,
                              nvr_stream_t stream);

/*
 * nvfp4_pack_weight -- load-time NVFP4 quantization of the gate weight.
 *
 * Source: "nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py",
 * NVFP4 gate section (BF16 gate weights are quantized and loaded into the
 * NVFP4 linear layer); "commit df05289", lm_head item (BF16 weight quantized
 * to NVFP4 at load time).
 *
 * The same arithmetic as nvfp4_quantize_act applied to W [N, D] with its own
 * global scale *w_gsa; scales always in the NVR_SF_TILED layout
 * (W_sf holds nvr_sf_bytes(N, D, NVR_SF_TILED) bytes).  Called once at load;
 * W_fp4, W_sf and w_gsa then stay resident and are passed to router_gate_topk.
 */
nvr_status nvfp4_pack_weight(const void* W, nvr_dtype dt, int64_t N, int64_t D,
                             uint8_t* W_fp4, uint8_t* W_sf, float* w_gsa,
                             void* workspace, size_t ws_bytes, nvr_stream_t stream);

/* Workspace bytes router_gate_topk / router_gate_logits need for up to
 * T_max tokens with this D, N and k (k is ignored by router_gate_logits). */
size_t router_gate_workspace_size(int64_t T_max, int64_t D, int64_t N, int k);

/*
 * router_gate_x_gsa_offset -- byte offset, inside a router workspace, of the
 * fp32 global scale gsa = max|x| / 2688 that the latest tensor-core
 * router_gate_topk / router_gate_logits call on that workspace computed for
 * its x ("commit df05289: dsv4/layers/grouped_linear.py", zero-sync fused
 * quantize section: the scale is produced and kept on the GPU, and other
 * kernels read it there).  The same for every T, D and N; 4-byte aligned.
 * Valid once that call's kernels have completed (stream order).  The decode
 * kernel (T <= 16) keeps its scale on chip and does not store it.
 */
size_t router_gate_x_gsa_offset(void);

/*
 * router_gate_topk -- the whole router call: quantize x, NVFP4 gate GEMM,
 * fused sigmoid / biased top-k / renormalise / scale epilogue.
 *
 * Sources: the three sections cited at the top of this file; the fused
 * single-kernel GEMM + router epilogue with a row-level top-k across
 * N-subtiles ("commit 04cf8ca", fused dispatch section; "commit e0f60b9",
 * fused decode kernel notes).
 *
 *   x            [T, D] activations (bf16 or fp32 per dt)
 *   W_fp4        [N, D/2] packed gate weight from nvfp4_pack_weight
 *   W_scales     its scale bytes (NVR_SF_TILED)
 *   w_gsa        its global scale (device fp32)
 *   bias         [N] fp32 score-correction bias added to the scores for
 *                selection only, or NULL for none (ignored in RAW mode)
 *   k            experts per token, 1 <= k <= min(16, N)
 *   routed_scaling  multiplies the renormalised weights
 *   flags        0 or NVR_FLAG_RAW_LOGITS, optionally with one kernel-choice
 *                flag (FORCE_TENSOR_CORE, FORCE_DECODE, SPLIT_K_2/4/8,
 *                SPLIT_N, STREAM) and, with a tensor-core choice or
 *                FORCE_DECODE, TEST_STALL
 *   out_ids      out [T, k] int32: expert ids, best first (key descending,
 *                equal keys: lower id first)
 *   out_w        out [T, k] fp32: routed_scaling * s_id / sum of the k
 *                selected sigmoid scores s (RAW: the selected logits)
 *   workspace    router_gate_workspace_size(T, D, N, k) bytes, zeroed once
 *
 * Launches per call (programmatic dependent launch chains several without
 * host involvement):
 *   - T <= 16 (decode): one kernel; for T >= 2 its CTAs form clusters of 4
 *     that share the staging and quantization of x through distributed
 *     shared memory.  Up to 256 experts CTA 0 selects: it polls the (key,
 *     score) words the other CTAs store into the workspace (bounded: a
 *     timeout records NVR_ERR_TIMEOUT in the status word) and puts them back
 *     to zero; wider heads end with the last CTA (an atomic ticket).
 *   - bf16 x, N <= 384: one kernel that takes max|x| itself (a bounded grid
 *     barrier in the workspace, or an exchange through distributed shared
 *     memory when the grid is one cluster), quantizes x inside the K-split
 *     GEMM and routes each tile's tokens from the fp32 partial logits
 *     (L2-resident workspace) after the tile's CTAs have met at a cluster
 *     barrier or, launched without clusters, at a workspace barrier.  When
 *     the grid cannot be resident at once (a forced split on a large T), an
 *     amax kernel runs first and the same kernel skips its own max|x| pass.
 *   - fp32 x, N <= 256: amax, quantize, K-split GEMM and a warp-per-token
 *     epilogue kernel.
 *   - N > 384 (fp32 x: N > 256), T <= 128: amax, quantize and the
 *     weight-streaming GEMM (the
 *     weight rows are the MMA's M, the tokens its N; each weight byte is read
 *     once), which routes from the logits in tensor memory and merges the
 *     CTAs' per-token lists in its last CTA.
 *   - N > 384 (fp32 x: N > 256), T > 128: amax, quantize and the N-split
 *     GEMM, which routes
 *     from the logits in tensor memory.
 */
nvr_status router_gate_topk(const void* x, nvr_dtype dt, int64_t T, int64_t D,
                            const uint8_t* W_fp4, const uint8_t* W_scales, const float* w_gsa,
                            int64_t N, const float* bias, int k, float routed_scaling,
                            uint32_t flags, int32_t* out_ids, float* out_w,
                            void* workspace, size_t ws_bytes, nvr_stream_t stream);

/*
 * router_gate_topk_noalloc -- router_gate_topk for callers that cannot
 * allocate device memory.  The pages have no counterpart to this entry
 * point; it exists for code whose host owns every device allocation (a plugin
 * handed only its input and output buffers) or that must not call an
 * allocator on its path, and so cannot pass a workspace.
 *
 * Same arguments and results as router_gate_topk, without the workspace.
 * It runs the single-launch decode kernel only (T <= 16 and a shape whose
 * per-CTA plan fits; otherwise NVR_ERR_UNSUPPORTED); flags may be 0 or
 * NVR_FLAG_RAW_LOGITS.  Its scratch (keys and scores of every (token, expert)
 * pair plus a ticket) lives in a fixed array of 224 KiB + 256 bytes in the
 * library's device memory, held by every GPU that loads the library until
 * the process exits.  That is the most the decode kernel's shared-memory plan
 * lets a call need (T * N * 8 bytes of keys and scores, the same bound); a
 * larger shape is refused by the plan (NVR_ERR_UNSUPPORTED).  It calls no
 * cudaMalloc/cudaFree.  Each call is one kernel launch on `stream` (the
 * ticket starts at zero and every launch leaves it at zero).
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) and caches it; make that first call before any
 *   stream capture.
 * - Every call shares the one array: calls whose kernels overlap on the GPU
 *   (different streams without ordering between them) race and give wrong
 *   results.  Order them on one stream.
 */
nvr_status router_gate_topk_noalloc(const void* x, nvr_dtype dt, int64_t T, int64_t D,
                                    const uint8_t* W_fp4, const uint8_t* W_scales,
                                    const float* w_gsa, int64_t N, const float* bias, int k,
                                    float routed_scaling, uint32_t flags, int32_t* out_ids,
                                    float* out_w, nvr_stream_t stream);

/*
 * router_hash_topk -- the hash router of the first MoE layers: each token's
 * experts are read from a token-id table, with no gate GEMM.
 *
 * Source: "nvfp4-megamoe-kernel commit df05289: dsv4/layers/grouped_linear.py",
 * hash-router item (tid2eid is an int32 lookup).  The page gives no weights;
 * with no gate scores the router's renormalise and scale steps see k equal
 * scores, so every selected expert weighs fl32(routed_scaling / k).
 *
 *   token_ids  [T] int32 token ids (device)
 *   tid2eid    [vocab, k] int32 table (device, row-major): row tid holds the
 *              k expert ids of token id tid, in output order
 *   n_experts  number of experts; 1 <= k <= min(16, n_experts)
 *   out_ids    out [T, k] int32: out_ids[t, j] = tid2eid[token_ids[t], j]
 *   out_w      out [T, k] fp32: routed_scaling / k
 * A token id outside [0, vocab) gives ids -1 and weights 0 for its row; a
 * table entry outside [0, n_experts) gives id -1 and weight 0 in its slot
 * (no out-of-bounds access in either case).  Host checks: NULL pointers,
 * T < 0, vocab < 1, k out of range (NVR_ERR_INVALID_ARG); pointers not 4-byte
 * aligned (NVR_ERR_ALIGNMENT).  One kernel, no workspace, no host sync;
 * T == 0 launches nothing (token_ids, out_ids and out_w may then be NULL).
 */
nvr_status router_hash_topk(const int32_t* token_ids, int64_t T, const int32_t* tid2eid, int64_t vocab,
                            int64_t n_experts, int k, float routed_scaling, int32_t* out_ids, float* out_w,
                            nvr_stream_t stream);

/*
 * nvfp4_linear -- an NVFP4 linear layer with a runtime activation scale:
 * out = quantize(x) . W^T, i.e. out[t, n] = sum_i xq[t, i] * wq[n, i] with
 * both operands dequantized (codes x block scales x global scales), fp32
 * accumulation on the tensor cores, stored as fp32 or bf16 (round to nearest
 * even).
 *
 * Source: "nvfp4-megamoe-kernel commit df05289: dsv4/layers/grouped_linear.py",
 * lm_head item (BF16 weight quantized to NVFP4 at load time, the production
 * NVFP4 GEMM, runtime gsa for the activation) and "commit 04cf8ca:
 * dsv4/layers/router.py", runtime-gsa section (the same runtime gsa in every
 * NVFP4 linear layer).
 *
 *   x        [T, D] activations (bf16 or fp32 per dt)
 *   W_fp4, W_scales, w_gsa   the weight [N, D] from nvfp4_pack_weight
 *   out      out [T, N] row-major, fp32 (out_dt NVR_F32) or bf16 (NVR_BF16),
 *            16-byte aligned
 *   workspace  nvfp4_linear_workspace_size(T, D, N) bytes, zeroed once
 * Launches: amax, quantize, then for T <= 128 the weight-streaming GEMM
 * (weight rows as the MMA's M, tokens as its N: each weight byte read once --
 * the lm_head shape at decode batch sizes), for more tokens the token-tiled
 * N-split GEMM.  Errors as for router_gate_topk.
 */
size_t nvfp4_linear_workspace_size(int64_t T_max, int64_t D, int64_t N);
nvr_status nvfp4_linear(const void* x, nvr_dtype dt, int64_t T, int64_t D, const uint8_t* W_fp4,
                        const uint8_t* W_scales, const float* w_gsa, int64_t N, void* out, nvr_dtype out_dt,
                        void* workspace, size_t ws_bytes, nvr_stream_t stream);

/*
 * nvfp4_moe_gemm -- the NVFP4 grouped expert GEMM fed by the router: every
 * routed (token, slot) pair is one row of expert ids[t, j]'s linear layer,
 *   y[t, j, n] = quantize(x)[t] . W_{ids[t,j]}[n]
 * with both operands dequantized (codes x block scales x global scales) and
 * fp32 accumulation on the tensor cores.
 *
 * Source: "nvfp4-megamoe-kernel commit df05289: dsv4/layers/grouped_linear.py"
 * (grouped NVFP4 linear: the groups' rows flattened into one tensor quantized
 * with one runtime global scale in one pass; expert offsets computed on the
 * GPU with no host synchronisation; pre-allocated buffers) and "commit
 * 04cf8ca: dsv4/layers/router.py", runtime-gsa section (Nvfp4GroupedLinear,
 * Nvfp4MoE).  x's global scale is max|x| / 2688 over x (each token is routed
 * k >= 1 times, so the flattened rows have the same maximum).
 *
 *   x          [T, D] activations (bf16 or fp32 per dt)
 *   ids        [T, k] int32 expert ids (router_gate_topk's out_ids); a pair
 *              whose id is outside [0, n_experts) gets a zero row
 *   W_fp4      [n_experts * N, D/2] the experts' packed weights stacked (expert
 *              e at rows e*N..), each from nvfp4_pack_weight of its [N, D]
 *   W_scales   their scale bytes, NVR_SF_TILED over the n_experts * N rows
 *              (expert e's nvr_sf_bytes(N, D, NVR_SF_TILED) bytes at
 *              e * nvr_sf_bytes(N, D, NVR_SF_TILED))
 *   w_gsa      [n_experts] the experts' global scales
 *   N          outputs per expert, a multiple of 128; n_experts <= 1024
 *   y          out [T, k, N] fp32 (y_dt NVR_F32) or bf16 (NVR_BF16)
 * x, ids, W_fp4, W_scales and y must be 16-byte aligned (NVR_ERR_ALIGNMENT).
 *   workspace  nvfp4_moe_gemm_workspace_size(T, D, n_experts, k) bytes,
 *              zeroed once
 * Four kernels, no host synchronisation: amax, a one-CTA routing kernel
 * (expert counts, 128-row padded segments, work units), a quantizer that
 * stores each token's codes and scales into its k expert-sorted rows, and the
 * grouped GEMM (each expert's weight tiles as the MMA's M, 128 of its token
 * rows as N).  The rows of one
 * expert are processed in an unspecified order; each output row is
 * independent of it, so results are deterministic.
 */
size_t nvfp4_moe_gemm_workspace_size(int64_t T_max, int64_t D, int64_t n_experts, int k);
nvr_status nvfp4_moe_gemm(const void* x, nvr_dtype dt, int64_t T, int64_t D, const int32_t* ids, int k,
                          int64_t n_experts, const uint8_t* W_fp4, const uint8_t* W_scales, const float* w_gsa,
                          int64_t N, void* y, nvr_dtype y_dt, void* workspace, size_t ws_bytes,
                          nvr_stream_t stream);

/*
 * nvfp4_moe_combine -- out[t, n] = sum_j w[t, j] * y[t, j, n], j in order
 * (fp32 fused multiply-adds): the router's weights (out_w) applied to the
 * grouped GEMM's rows.  y [T, k, N] fp32 or bf16 per y_dt, w [T, k] fp32,
 * out [T, N] fp32; N a multiple of 4; y and out 16-byte aligned.  One kernel,
 * no workspace.  No counterpart on the pages beyond the weighted sum the
 * router's weights exist for.
 */
nvr_status nvfp4_moe_combine(const void* y, nvr_dtype y_dt, int64_t T, int k, int64_t N, const float* w,
                             float* out, nvr_stream_t stream);

/*
 * router_gate_logits -- test hook: the same quantization and gate GEMM as
 * router_gate_topk, writing the fp32 logits [T, N] (row-major,
 * logit = acc * gsa_x * gsa_w) instead of the epilogue's outputs.  Used to
 * check the GEMM on its own and to measure what writing logits to memory
 * costs.  flags: 0 or one kernel-choice flag (FORCE_TENSOR_CORE,
 * FORCE_DECODE, SPLIT_K_2/4/8, SPLIT_N, STREAM); RAW_LOGITS and TEST_STALL
 * are invalid here.  Workspace as for router_gate_topk.
 */
nvr_status router_gate_logits(const void* x, nvr_dtype dt, int64_t T, int64_t D,
                              const uint8_t* W_fp4, const uint8_t* W_scales, const float* w_gsa,
                              int64_t N, uint32_t flags, float* logits, void* workspace,
                              size_t ws_bytes, nvr_stream_t stream);

/*
 * nvr_set_profile_events -- measurement hook (no counterpart on the pages; it
 * serves the benchmark's per-kernel roofline).  When `events` is not NULL,
 * every later call of nvfp4_quantize_act, nvfp4_pack_weight,
 * router_gate_topk and router_gate_logits records events[2*i] just before and
 * events[2*i+1] just after its i-th kernel launch (i < n_pairs), on the call's
 * stream; launches beyond n_pairs are not bracketed.  The events are
 * cudaEvent_t handles created by the caller.  Recording an event between two
 * launches removes their programmatic overlap, so time whole calls with the
 * hook off.  NULL (or n_pairs <= 0) turns the hook off.  Process-wide
 * setting; not thread-safe.
 */
nvr_status nvr_set_profile_events(void* const* events, int n_pairs);

/*
 * nvr_read_device_status -- copy the workspace status word to *out (blocking
 * read on `stream`; do not call during stream capture).  NVR_OK unless a
 * device-side bounded wait timed out (NVR_ERR_TIMEOUT).
 */
nvr_status nvr_read_device_status(const void* workspace, nvr_stream_t stream, nvr_status* out);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_ROUTER_H */
