// gemm_fused.cu -- the router for up to 384 experts on bf16 activations in one
// launch: max|x| over the CTAs' own x boxes and a grid barrier (or, when the
// grid cannot be resident at once, the amax kernel launched before), then the
// runtime NVFP4 quantization of x inside a K-split tensor-core GEMM and the
// router epilogue in the same kernel, so the quantized activations never
// exist in memory and the logits only pass through L2 (sm_103a).
//
// Source: "nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py"
// (runtime gsa = max|x| / 2688, NVFP4 activations and gate weight, gate GEMM
// on Blackwell tensor cores, the single-kernel GEMM + fused router epilogue)
// and "commit e0f60b9: dsv4/kernels/router/__init__.py" (activation_topk).
// Quantization arithmetic as in the standalone quantizer (quant_block16):
// y = RN(x / gsa), sy = RN(max|y| / 6), E4M3 scale, E2M1 codes of
// RN(y / scale) with the input's sign; identical codes and scale bytes,
// reached by table lookups and bracketing products (quant_rows_bracket) with
// an exact pass over the rare rows near a rounding boundary.
//
// A token tile of 128 (or 112) rows is split along K over S CTAs (S = 1 to
// 16, a power of two) that form one thread-block cluster, or, in a grid the
// device holds at once without clusters, meet at a barrier in the workspace
// (tile_barrier) before routing.  Per CTA (rank r, 576 threads):
//   warp 0      TMA producer.  With the in-kernel max|x| it first streams the
//               CTA's own x boxes in reverse K order into a 5- or 6-slot
//               ring laid over the other rings (the second pass then starts
//               on the boxes read last, still in L2 where x is larger than
//               L2), then per stage of 256 K-elements two bf16 x boxes (128
//               rows x 128 elements, 32 KB each) into a 3-slot ring, and the
//               W tile (128 kNT rows x 128 bytes, 128-byte swizzle) with its
//               scale slabs into a 2-deep ring (kNT = 3: 1-deep);
//   warps 2-17  quantizers (quant_box): warps 2-9 take the stage's first x
//               box, warps 10-17 its second, 1/8 of the box rows per warp;
//               they write the E2M1 codes into the A tile (128-byte swizzle,
//               the layout TMA would have produced) and the scale bytes into
//               the stage's scale atoms; the A tile is double-buffered and
//               the warps synchronise only through mbarriers (a warp may run
//               about a stage ahead of another);
//   warp 1      MMA issuer: once all sixteen quantizer warps have filled the A
//               slot, copies the stage's x and W scale atoms into tensor
//               memory (tcgen05.cp, in order with the MMAs on the otherwise
//               idle tensor pipe) and issues one tcgen05.mma.kind::mxf4nvf4
//               (M=128, N=128 or 256, K=64) per 64-element K step into one
//               fp32 accumulator (kNT = 3, 257-384 experts: an N=256 and an
//               N=128 MMA into columns 0-255 and 256-383);
//   warps 2-17  after the last MMA: the fp32 partial (128 x 128 kNT) goes from
//               tensor memory through shared memory (TMA stores) to partial
//               plane r of the workspace (L2); after a
//               cluster (or tile) barrier each CTA routes its own 128/S tokens
//               from the S planes, one warp per token (TokenRouter,
//               nvr_splitk.cuh).
// The quantizers are bound by the integer pipe: sixteen warps reach the same
// throughput per SM as eight, but leave half as many rows per warp for the
// epilogue.  Tensor memory: accumulator at columns 0 .. 128 kNT - 1; scales of
// A slot a at 128 kNT + (16 + 16 kNT) a (x: 4 columns per K step, W: 4 kNT).
#include <type_traits>

#include "nvr_splitk.cuh"

namespace nvr {

namespace {

constexpr int kFXBox = 128 * 128 * 2;               // 128 rows x 128 bf16
constexpr int kFASlots = 2;
constexpr int kFACodes = 128 * 128;                 // 128 token rows x 128 bytes of codes
constexpr int kFASfa = 4 * 512;                     // 4 scale atoms
constexpr int kFASlot = kFACodes + kFASfa;
constexpr int kFARing = kFASlots * kFASlot;
constexpr int kFXSlots = 3;
constexpr int kFXRing = kFXSlots * kFXBox;
constexpr int kFByteTab = 2560;                     // scale bytes of bf16 block maxima (amax down ~20 binades)
constexpr int kFFixQ = 256;                         // exact-pass queue entries per quantizer warp and box (>= 32 x groups)
constexpr int kFQWarps = 16;                        // quantizer warps: 8 per x box, both boxes of a stage at once
constexpr int kFQThreads = 32 * kFQWarps;
constexpr int kFTables = 1024 + 1024 + kFByteTab + kFQWarps * kFFixQ * 2;   // s_scale, s_cc, s_byte, s_fixq
constexpr int kFThreads = 64 + kFQThreads;
constexpr int kFChunk = 32768;
// The shared-memory plan for heads of up to 128 kNT experts (kNT = 2: up to
// 256, kNT = 3: up to 384).  The W tile of a stage holds 128 kNT rows x 128
// bytes and kNT x 4 scale atoms; with kNT = 3 one stage is buffered (a W
// tile comes from L2 in about 1 us while the quantizers take longer over a
// stage), else two.  The max|x| pass streams the CTA's x boxes (up to 32 KB
// each) through a ring over the W, x and A rings (all idle until the pass
// ends).
template <int kNT>
struct FusedCfg {
  static_assert(kNT == 2 || kNT == 3, "up to 256 or 384 experts");
  static constexpr int kStagesW = kNT == 3 ? 1 : 2;
  static constexpr int kWTile = 128 * kNT * 128;
  static constexpr int kSfb = kNT * 4 * 512;
  static constexpr int kWStage = kWTile + kSfb;
  static constexpr int kWRing = kStagesW * kWStage;
  static constexpr int kChunkSlots = (kWRing + kFXRing + kFARing) / kFChunk < 6 ? (kWRing + kFXRing + kFARing) / kFChunk : 6;
  static constexpr int kSmem = kWRing + kFXRing + kFARing + kFTables + 512 /*barriers*/ + 1024 /*align*/;
  // tensor memory: the accumulator at columns 0 .. 128 kNT - 1, then per A
  // slot the x scales (4 columns per K step) and the W scales (4 kNT)
  static constexpr int kScaleCol = 128 * kNT;
  static constexpr int kScaleSlot = 16 + 16 * kNT;
  static_assert(kScaleCol + kFASlots * kScaleSlot <= 512, "tensor memory");
  static_assert(kWStage % 1024 == 0 && kFASlot % 1024 == 0 && kFXBox % 1024 == 0, "1024-byte aligned tiles");
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert(kChunkSlots >= 4, "the max|x| ring");
};
static_assert(16 * 4096 <= kFXRing, "store staging fits the x ring");
// A token tile has kRows = 128 or 112 rows (the kernel is instantiated for
// both): each of the eight quantizer warps of a box takes kRows / 8 rows, that
// is kRows / 16 row pairs, quantized as one group (their chains interleave).
// With 112 the MMA's last 16 accumulator rows are junk and never stored.

struct FusedParams {
  CUtensorMap tmap_x;          // bf16 activations [T, D], box 128 x 128, no swizzle
  CUtensorMap tmap_b;          // W codes [N, D/2] uint8, box 128 bytes x 128 n_groups rows (kNT = 3: 128)
  CUtensorMap tmap_p;          // partial rows [S][T][128 kNT] fp32, box 32 x 16 x 1, 128-byte swizzle
  float* qrec;                 // quantizer record {gsa, 1/gsa, mode, amax}: from the amax kernel, or
                               // published by this kernel's last CTA when amax_sync is set
  uint32_t* amax_sync;         // in-kernel amax: 5 workspace words (grid_amax), or null
  uint32_t* tile_sync;         // with amax_sync: the tile barriers' arrival counters [2][kMaxFlatTiles]
  int flat;                    // launch without clusters: a tile's CTAs meet at tile_barrier
  float* gsa_out;              // in-kernel amax: x's global scale (also x_gsa)
  const uint8_t* sfb;          // W scales, tile layout
  float* partials;             // [S][T][256] fp32 partial logits (workspace)
  int T, D, N, n_groups, S;   // n_groups: 128-expert groups of the head (1 .. kNT)
  // router epilogue
  const float* x_gsa;
  const float* w_gsa;
  const float* bias;           // [N] or null
  int k, raw;
  float routed_scaling;
  int32_t* out_ids;
  float* out_w;
  float* logits;               // logits mode: write [T, N] logits instead of the top-k
  uint32_t* status;
  int test_stall;              // test hook: the MMA issuer issues nothing
};

__device__ __forceinline__ void st_shared_u32(uint8_t* p, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" :: "r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_u8(uint8_t* p, uint32_t v) {
  asm volatile("st.shared.u8 [%0], %1;" :: "r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Grid-wide max |x| bits, for one thread per CTA, over 5 workspace words:
// sync[0..1] the maximum and sync[2..3] the arrivals of calls of even / odd
// generation, sync[4] the generation.  A CTA folds its max into its
// generation's slot and arrives (a release increment, nothing returned);
// all then wait (acquire, bounded) until every CTA has arrived -- nobody has
// to answer anybody -- and read the complete max.  CTA 0 then bumps the
// generation for the next call (every CTA of this call read it before
// arriving: `gen`, read before the CTA's max|x| pass, so that no round trip
// for it lies between the last CTA's pass and the barrier -- 0.3 us earlier
// at T = 4096).  Each call zeroes the other generation's words at its start
// (the call that used them has completed).  All CTAs of the grid must be
// resident.  Measured and not kept: per-CTA maximum words with a presence
// bit, every CTA reading all of them instead of an arrival counter (no
// counter, no second read): the 148 pollers' reads contend at the L2 and the
// barrier ended 1.9 us later.
__device__ bool grid_amax(uint32_t* sync, uint32_t gen, uint32_t cta_max, uint32_t n_ctas, uint32_t& amax_bits,
                          uint64_t deadline, volatile int* abort_flag) {
  const uint32_t par = gen & 1u;
  asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" :: "l"(sync + par), "r"(cta_max) : "memory");
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(sync + 2 + par) : "memory");
  while (ld_acquire_gpu(sync + 2 + par) < n_ctas)
    if (*abort_flag || globaltimer_ns() > deadline) return false;
  if (blockIdx.x == 0) sync[4] = gen + 1u;
  amax_bits = ld_acquire_gpu(sync + par);
  return true;
}

// Barrier of the n CTAs of one token tile, for one thread per CTA, on one
// arrival counter in the workspace: a release increment, then acquire reads
// until all n have arrived -- no CTA has to answer another, so the barrier
// costs one trip to L2 and back after the last arrival.  The partial rows the
// CTA's threads stored before a __syncthreads are visible to the other CTAs
// after theirs.  Calls alternate between two counter sets by the parity of
// the grid barrier's generation (the same in every CTA of a call); each call
// zeroes the other set's counter of its tile for the next call (the call that
// used it has completed; every call with the in-kernel amax does this, with
// or without clusters).  The n CTAs must be resident together.
__device__ bool tile_barrier(uint32_t* count, uint32_t n, uint64_t deadline, volatile int* abort_flag) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(count) : "memory");
  while (ld_acquire_gpu(count) < n)
    if (*abort_flag || globaltimer_ns() > deadline) return false;
  return true;
}

// Quantize kG rows of one stage, 8 bf16 values (half of a 16-element block;
// the other half sits in lane ^ 1) per row and lane.  The rows are
// independent and the code is branch-free, so their dependency chains
// interleave.  kMode: 1 = division shortcut (gsa and 1/gsa in [2^-80, 2^80]),
// 2 = IEEE division.  Writes each row's 4 packed code bytes to codes[] and the
// block's E4M3 scale byte to bytes[].  s_scale[b] = (dec(b), RN(1/dec(b))).
template <int kMode, int kG>
__device__ __forceinline__ void quant_rows(const uint4 (&v)[kG], const QuantScale& qs, const float2* s_scale,
                                           uint32_t (&codes)[kG], uint32_t (&bytes)[kG]) {
  const float r6 = 0.16666667163372039794921875f;       // RN(1/6)
  float x[kG][8];
  float mx[kG];
#pragma unroll
  for (int i = 0; i < kG; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[i][2 * j] = __uint_as_float(w[j] << 16);
      x[i][2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
    // max |x| on the bf16 bit patterns (integer pipe; exact)
    mx[i] = __uint_as_float(absmax_bits16B<true>(v[i]));
  }
#pragma unroll
  for (int i = 0; i < kG; ++i) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xFFFFFFFFu, mx[i], 1));
  const uint64_t ng2 = f2_pack(-qs.gsa, -qs.gsa), rg2 = f2_pack(qs.rgsa, qs.rgsa);
#pragma unroll
  for (int i = 0; i < kG; ++i) {
    // max|y| = RN(max|x| / gsa): rounding is monotone
    const float ymax = kMode == 1 ? div_rn(mx[i], qs.gsa, qs.rgsa) : __fdiv_rn(mx[i], qs.gsa);
    bytes[i] = e4m3_byte(div_rn_short(ymax, 6.0f, r6));
    const float2 sr = s_scale[bytes[i]];
    const uint64_t ns2 = f2_pack(-sr.x, -sr.x), rs2 = f2_pack(sr.y, sr.y);
    float z[8];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const uint64_t y = kMode == 1 ? div_rn2(f2_pack(x[i][j], x[i][j + 1]), ng2, rg2)
                                    : f2_pack(__fdiv_rn(x[i][j], qs.gsa), __fdiv_rn(x[i][j + 1], qs.gsa));
      const uint64_t q = div_rn2_short(y, ns2, rs2);
      z[j] = f2_lo(q);
      z[j + 1] = f2_hi(q);
    }
    const uint32_t c = e2m1_pack8(z[0], z[1], z[2], z[3], z[4], z[5], z[6], z[7]) |
                       bf16x8_sign_nibbles(v[i].x, v[i].y, v[i].z, v[i].w);
    codes[i] = bytes[i] ? c : 0u;                       // a zero scale byte: all codes 0
  }
}

// Mode-1 quantizer of kG rows by bracketing products: the scale bytes of
// quant_rows<1, kG> and, wherever mism[i] is 0, its codes, at a quarter of its
// multiply-adds.
//   scale byte: a function of the block's max|x| alone (monotone), looked up
//     in s_byte[], which holds it for every bf16 max from amax down by 2559
//     steps (about 20 binades; anything smaller has a zero byte, as has the
//     last entry);
//   code: with c = RN(1/gsa) * RN(1/s) (rounded) and c_lo/hi = c (1 -/+ 2^-20)
//     (rounded), P_lo/hi = RN(x c_lo/hi) lie on both sides of the exact
//     q = RN(RN(x / gsa) / s): each of them is within 5 ulp of x / (gsa s) and
//     q within 2, far inside the 2^-20 margin (16 ulp).  E2M1 rounding is
//     monotone, so where the two codes agree the exact code equals them.
//     Where they differ (q within ~2^-20 of a rounding boundary, e.g. an exact
//     tie), mism[i] != 0 and the row's codes must be recomputed exactly
//     (quant_cell_exact).
//   sign of zero: an element that rounds to zero gets code 0x0 whatever its
//     sign (the conversion drops it; the standalone quantizer restores 0x8).
//     A zero code adds +-0 to the tensor-core dot product, which changes
//     nothing but the sign of an all-zero sum, and sigmoid(+0) = sigmoid(-0):
//     the router's scores, ids and weights are the same.
// s_cc[b] = (c_lo, c_hi) of scale byte b (zero for byte 0).
__device__ __forceinline__ uint32_t bf16x2_max_abs(uint32_t a, uint32_t b) {
  uint32_t d;   // magnitude max(|a|, |b|) per half (the sign bit is the xor of the inputs')
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

template <int kG>
__device__ __forceinline__ void quant_rows_bracket(const uint4 (&v)[kG], const uint8_t* s_byte, uint32_t amax_b16,
                                                   const float2* s_cc, uint32_t (&codes)[kG],
                                                   uint32_t (&bytes)[kG], uint32_t (&mism)[kG]) {
#pragma unroll
  for (int i = 0; i < kG; ++i) {
    // the block's max |x| (bf16 magnitude bits): this lane's 8 values, then
    // its partner's, then the two halves (finite inputs: mode 1)
    uint32_t m = bf16x2_max_abs(bf16x2_max_abs(v[i].x, v[i].y), bf16x2_max_abs(v[i].z, v[i].w));
    m = bf16x2_max_abs(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = bf16x2_max_abs(m, __byte_perm(m, 0u, 0x1032));
    // s_byte[d] holds the byte of the block max with bf16 bits amax - d
    bytes[i] = s_byte[min(amax_b16 - (m & 0x7FFFu), static_cast<uint32_t>(kFByteTab - 1))];
  }
#pragma unroll
  for (int i = 0; i < kG; ++i) {
    const float2 cc = s_cc[bytes[i]];
    const uint64_t lo2 = f2_pack(cc.x, cc.x), hi2 = f2_pack(cc.y, cc.y);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    float a[8], b[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint64_t xp = f2_pack(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u));
      const uint64_t pl = f2_mul(xp, lo2), ph = f2_mul(xp, hi2);
      a[2 * j] = f2_lo(pl); a[2 * j + 1] = f2_hi(pl);
      b[2 * j] = f2_lo(ph); b[2 * j + 1] = f2_hi(ph);
    }
    // a zero scale byte has zero multipliers: its codes come out zero
    codes[i] = e2m1_pack8(a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7]);
    mism[i] = codes[i] ^ e2m1_pack8(b[0], b[1], b[2], b[3], b[4], b[5], b[6], b[7]);
  }
}

// Exact mode-1 codes of one row's 8 values (half a block) with a known
// nonzero scale byte: y = RN(x / gsa) and q = RN(y / s) by the division
// shortcuts, as in quant_rows<1, 1> (zero codes unsigned, as in
// quant_rows_bracket).
__device__ __forceinline__ uint32_t quant_cell_exact(const uint4 v, uint32_t byte, const QuantScale& qs,
                                                     const float2* s_scale) {
  const float2 sr = s_scale[byte];
  const uint64_t ng2 = f2_pack(-qs.gsa, -qs.gsa), rg2 = f2_pack(qs.rgsa, qs.rgsa);
  const uint64_t ns2 = f2_pack(-sr.x, -sr.x), rs2 = f2_pack(sr.y, sr.y);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float z[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint64_t xp = f2_pack(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u));
    const uint64_t q = div_rn2_short(div_rn2(xp, ng2, rg2), ns2, rs2);
    z[2 * j] = f2_lo(q);
    z[2 * j + 1] = f2_hi(q);
  }
  return e2m1_pack8(z[0], z[1], z[2], z[3], z[4], z[5], z[6], z[7]);
}

// Per-call quantizer constants and the shared-memory tables built from them.
struct QuantTables {
  QuantScale qs;
  const float2* s_scale;     // [128] (dec(b), RN(1/dec(b)))
  const float2* s_cc;        // [128] bracketing multipliers of byte b
  const uint8_t* s_byte;     // [kFByteTab] scale byte of a bf16 block max
  uint32_t amax_b16;         // bf16 bits of amax: s_byte[d] is for amax_b16 - d
};

// Stores of one 4-row group: each row's 4 code bytes into the A slot's
// 128-byte swizzled layout (the one TMA would produce; box hs fills chunks
// 4hs..4hs+3 of a row) and each block's scale byte into the slot's scale atoms.
template <int G>
__device__ __forceinline__ void store_group(uint8_t* ac, uint8_t* asf, int hs, int row0, int sub, int l16,
                                            const uint32_t (&codes)[G], const uint32_t (&bytes)[G]) {
  const int j = 4 * hs + (l16 >> 2);                     // 16-byte chunk of the code row
  const int c = 8 * hs + (l16 >> 1);                     // 16-element block of the stage
#pragma unroll
  for (int i = 0; i < G; ++i) {
    const int r = row0 + 2 * i + sub;
    // codes: 4 bytes at chunk j ^ (r % 8), offset 4 * (l16 % 4)
    st_shared_u32(ac + r * 128 + (((j ^ (r & 7)) << 4) | ((l16 & 3) << 2)), codes[i]);
    // scale byte of block c: atom c/4, line r % 32, group (r/32) % 4, byte c % 4
    if (!(l16 & 1))
      st_shared_u8(asf + 512 * (c >> 2) + 16 * (r & 31) + 4 * ((r >> 5) & 3) + (c & 3), bytes[i]);
  }
}

// One quantizer warp's share of an x box (128 rows x 128 bf16, row stride 256
// bytes): its 16 rows, two per instruction (lanes 0-15 and 16-31), lane l16
// holding 8 values -- half of a 16-element block, whose other half sits in
// lane ^ 1.  Rows at or past row_end are skipped, eight at a time.
// fixq: this warp's exact-pass queue.  Mode 1 runs the bracketing quantizer
// and then the exact pass over the queued rows; the other modes (IEEE
// division, or gsa == 0: all codes zero) run in a loop of their own, so that
// the hot loop holds no other code.
template <int kRows>
__device__ __forceinline__ void quant_box(const uint8_t* xb, uint8_t* ac, uint8_t* asf, int hs, int qw, int lane,
                                          int row_end, const QuantTables& tb, uint16_t* fixq) {
  constexpr int kFRowsPerWarp = kRows / 8, kFGroup = kRows / 16;
  static_assert(kFGroup <= 8, "row pairs fit the 3-bit queue field");
  const QuantScale& qs = tb.qs;
  const int sub = lane >> 4, l16 = lane & 15;
  if (qs.mode != 1) {
#pragma unroll 1
    for (int g = 0; g < kFRowsPerWarp / 2; ++g) {
      if (qw * kFRowsPerWarp + 2 * g >= row_end) break;
      uint4 v[1];
      v[0] = ld_shared_v4(xb + (qw * kFRowsPerWarp + 2 * g + sub) * 256 + 16 * l16);
      uint32_t codes[1] = {0u}, bytes[1] = {0u};
      if (qs.mode == 2) quant_rows<2, 1>(v, qs, tb.s_scale, codes, bytes);
      store_group<1>(ac, asf, hs, qw * kFRowsPerWarp + 2 * g, sub, l16, codes, bytes);
    }
    return;
  }
  uint32_t n_fix = 0;                                      // queued rows (warp-uniform)
#pragma unroll
  for (int g = 0; g < kFRowsPerWarp / 2; g += kFGroup) {
    // rows past T only feed accumulator rows that are never stored: a group
    // that starts past T is skipped (warp-uniform)
    if (qw * kFRowsPerWarp + 2 * g >= row_end) break;
    uint4 v[kFGroup];
#pragma unroll
    for (int i = 0; i < kFGroup; ++i)
      v[i] = ld_shared_v4(xb + (qw * kFRowsPerWarp + 2 * (g + i) + sub) * 256 + 16 * l16);
    uint32_t codes[kFGroup], bytes[kFGroup], mism[kFGroup];
    quant_rows_bracket<kFGroup>(v, tb.s_byte, tb.amax_b16, tb.s_cc, codes, bytes, mism);
    // lanes with rows whose bracketing codes differ go to the exact pass:
    // entry = lane (5 bits) | first row pair of the group (3 bits) << 5 |
    // mask of the group's rows to redo << 8
    uint32_t redo = 0;
#pragma unroll
    for (int i = 0; i < kFGroup; ++i) redo |= (mism[i] != 0u ? 1u : 0u) << i;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, redo != 0u);
    if (redo) fixq[n_fix + __popc(bal & ((1u << lane) - 1u))] = static_cast<uint16_t>(lane | (g << 5) | (redo << 8));
    n_fix += __popc(bal);
    store_group<kFGroup>(ac, asf, hs, qw * kFRowsPerWarp + 2 * g, sub, l16, codes, bytes);
  }
  if (n_fix) {
    // exact pass over the queued lanes, one lane per entry: every flagged row
    // of the entry's group, its block's scale byte found again from both
    // halves of the block; the box is still in shared memory (the caller
    // releases it afterwards)
    __syncwarp();
    for (uint32_t e0 = 0; e0 < n_fix; e0 += 32) {
      if (e0 + lane < n_fix) {
        const uint32_t ent = fixq[e0 + lane];
        const int ln = ent & 31, l = ln & 15;
        const int row_pair0 = static_cast<int>((ent >> 5) & 7u);
        for (uint32_t redo = ent >> 8; redo; redo &= redo - 1u) {
          const int r = qw * kFRowsPerWarp + 2 * (row_pair0 + __ffs(redo) - 1) + (ln >> 4);
          const uint4 v = ld_shared_v4(xb + r * 256 + 16 * l);
          const uint4 w = ld_shared_v4(xb + r * 256 + 16 * (l ^ 1));
          uint32_t m = bf16x2_max_abs(bf16x2_max_abs(bf16x2_max_abs(v.x, v.y), bf16x2_max_abs(v.z, v.w)),
                                      bf16x2_max_abs(bf16x2_max_abs(w.x, w.y), bf16x2_max_abs(w.z, w.w)));
          m = bf16x2_max_abs(m, __byte_perm(m, 0u, 0x1032));
          const uint32_t byte = tb.s_byte[min(tb.amax_b16 - (m & 0x7FFFu), static_cast<uint32_t>(kFByteTab - 1))];
          const int j = 4 * hs + (l >> 2);
          st_shared_u32(ac + r * 128 + (((j ^ (r & 7)) << 4) | ((l & 3) << 2)),
                        quant_cell_exact(v, byte, qs, tb.s_scale));
        }
      }
    }
  }
}

template <int kRows, int kNT>
__global__ void __launch_bounds__(kFThreads, 1)
fused_qgemm_kernel(const __grid_constant__ FusedParams p) {
  using C = FusedCfg<kNT>;
  constexpr int kFStagesW = C::kStagesW, kFWTile = C::kWTile, kFWStage = C::kWStage, kFWRing = C::kWRing;
  constexpr int kFChunkSlots = C::kChunkSlots;
  constexpr int kFRowsPerWarp = kRows / 8;
  constexpr uint32_t kBoxBytes = 128u * kRows * 2u;  // one bf16 x box: kRows rows x 128 elements
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wring = smem;
  uint8_t* xring = wring + kFWRing;
  uint8_t* aring = xring + kFXRing;
  float2* s_scale = reinterpret_cast<float2*>(aring + kFARing);        // [128] (dec(b), RN(1/dec(b)))
  float2* s_cc = s_scale + 128;                                         // [128] (c_lo, c_hi) of byte b
  uint8_t* s_byte = reinterpret_cast<uint8_t*>(s_cc + 128);             // [kFByteTab] scale byte of a block max
  uint16_t* s_fixq = reinterpret_cast<uint16_t*>(s_byte + kFByteTab);   // [16][kFFixQ] rows for the exact pass
  uint64_t* full_w = reinterpret_cast<uint64_t*>(s_fixq + kFQWarps * kFFixQ);
  uint64_t* empty_w = full_w + kFStagesW;
  uint64_t* full_x = empty_w + kFStagesW;
  uint64_t* empty_x = full_x + kFXSlots;
  uint64_t* a_empty = empty_x + kFXSlots;
  uint64_t* q_done = a_empty + kFASlots;                               // [kFASlots]
  uint64_t* acc_full = q_done + kFASlots;
  uint64_t* amax_mbar = acc_full + 1;           // one-cluster grids: the S CTAs' maxima have landed
  uint64_t* full_c = amax_mbar + 1;             // [kFChunkSlots] max|x| pass ring
  uint64_t* empty_c = full_c + kFChunkSlots;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(empty_c + kFChunkSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  // producer: ring slots with a fill in flight and the parity of their latest fill
  uint32_t filled_w = 0, bits_w = 0, filled_x = 0, bits_x = 0, filled_c = 0, bits_c = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x / p.S;
  const int rank = blockIdx.x - m_tile * p.S;
  const int KB = p.D / kBlock;
  const int n_st = (KB + 15) / 16;                   // stages of 256 K-elements
  const int st0 = (rank * n_st) / p.S;
  const int my_st = ((rank + 1) * n_st) / p.S - st0;
  // the max|x| pass reads the CTA's own 2 my_st x boxes, in reverse K order
  const int n_chunks = 2 * my_st;                    // boxes of the max|x| pass

  if (threadIdx.x == 0) {
    for (int s = 0; s < kFStagesW; ++s) { mbar_init(full_w + s, 1); mbar_init(empty_w + s, 1); }
    for (int s = 0; s < kFXSlots; ++s) { mbar_init(full_x + s, 1); mbar_init(empty_x + s, 8); }
    for (int a = 0; a < kFASlots; ++a) {
      mbar_init(a_empty + a, 1);
      mbar_init(q_done + a, kFQWarps);
    }
    mbar_init(acc_full, 1);
    mbar_init(amax_mbar, p.S);
    for (int c = 0; c < kFChunkSlots; ++c) { mbar_init(full_c + c, 1); mbar_init(empty_c + c, kFQWarps); }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&p.tmap_x);
    tma_prefetch_map(&p.tmap_b);
    tma_prefetch_map(&p.tmap_p);
  }
  if (threadIdx.x < 128) {
    const uint32_t b = threadIdx.x;
    const bool ok = b >= 1 && b <= 126;
    s_scale[b] = make_float2(ok ? e4m3_value(b) : 0.0f, ok ? __frcp_rn(e4m3_value(b)) : 0.0f);
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // A grid of one cluster exchanges the CTAs' maxima through distributed
  // shared memory: every CTA must run, its mbarrier initialised, first.
  const bool one_cluster = p.amax_sync && !p.flat && gridDim.x == static_cast<unsigned>(p.S) && p.S > 1;
  if (one_cluster) cluster_sync_all();
  // the amax kernel before us (programmatic launch) must have finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Barrier words: this call uses those of the grid barrier's generation
  // parity (the same for every CTA until all have arrived there) and zeroes
  // the other parity's -- the grid barrier's maximum and arrivals and the
  // whole set of tile-barrier counters -- for the next call.
  uint32_t* tile_count = nullptr;
  if (p.amax_sync && warp == 0) {
    const uint32_t par = ld_acquire_gpu(p.amax_sync + 4) & 1u;
    tile_count = p.tile_sync + par * kMaxFlatTiles + m_tile;
    uint32_t* other = p.tile_sync + (par ^ 1u) * kMaxFlatTiles;
    for (int i = blockIdx.x * 32 + lane; i < kMaxFlatTiles; i += gridDim.x * 32) other[i] = 0u;
    if (blockIdx.x == 0 && lane == 0) {
      p.amax_sync[par ^ 1u] = 0u;
      p.amax_sync[2 + (par ^ 1u)] = 0u;
    }
  }
  // The next kernel of the stream may launch now; it waits for this grid to
  // complete before it reads anything.
  asm volatile("griddepcontrol.launch_dependents;");
  const uint64_t deadline = globaltimer_ns() + 1000000000ull;   // 1 s

  bool acc_ok = true;     // quantizer warps: the accumulator is complete
  TokenRouterT<kNT> rt;   // quantizer warps: the epilogue's per-lane state
  float gscale = 0.0f;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int wst = 0;
    uint32_t wph = 0;
    bool ok = true;
    int xi = 0;                                        // x boxes issued so far
    // With the in-kernel amax, x streams twice: the CTA's boxes for the max
    // (one pass over x in HBM), then again for the GEMM.  The first pass
    // takes them in reverse K order, so that the second starts on the boxes
    // read last: where x is larger than L2 (T = 16384: 235 MB) those are the
    // ones still there.  The second pass starts as soon as every box of the
    // first has been consumed (the max-pass ring overlays the other rings),
    // its loads overlapping the grid barrier.
    if (p.amax_sync) {
      for (int c = 0; c < n_chunks; ++c) {
        const int cs = c % kFChunkSlots;
        const uint32_t cph = (c / kFChunkSlots) & 1;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty_c + cs, cph ^ 1u, deadline, abort_flag))) {
          ok = false;
          break;
        }
        if (elect_one()) {
          const int bi = n_chunks - 1 - c;             // box hs = bi % 2 of stage st0 + bi / 2
          mbar_arrive_expect_tx(full_c + cs, kBoxBytes);
          tma_load_2d(smem + cs * kFChunk, &p.tmap_x, (st0 + bi / 2) * 256 + (bi & 1) * 128, m_tile * kRows,
                      full_c + cs);
        }
        __syncwarp();
        filled_c |= 1u << cs;
        bits_c = (bits_c & ~(1u << cs)) | (cph << cs);
      }
      for (int cs = 0; cs < kFChunkSlots && ok; ++cs)
        if ((filled_c >> cs) & 1u)
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(empty_c + cs, (bits_c >> cs) & 1u, deadline, abort_flag));
    }
    if constexpr (kNT == 3) {
      // kNT = 3 (one W stage): the x boxes and the W tiles are issued
      // independently, each as soon as its ring slot is free, so that the x
      // ring runs as far ahead as its slots allow while a W tile waits for the
      // MMAs that free its slot (issuing the next stage's boxes only after the
      // W slot -- the order below for kNT = 2 -- left the quantizer warps
      // waiting on x: adversarial batch 146.0 -> 139.6 us).  Non-blocking
      // tests, with a short sleep when neither ring has room.
      const int nx = 2 * my_st;
      int wi = 0;                                        // W stages issued so far
      uint64_t polls = 0;
      while (ok && (xi < nx || wi < my_st)) {
        bool progressed = false;
        if (xi < nx) {
          const int xs = xi % kFXSlots;
          const uint32_t xph = (xi / kFXSlots) & 1;
          if (__all_sync(0xFFFFFFFFu, mbar_test_wait(empty_x + xs, xph ^ 1u))) {
            const int ks = st0 + xi / 2, hs = xi & 1;     // box hs of stage ks (past D or T: zeros)
            if (elect_one()) {
              mbar_arrive_expect_tx(full_x + xs, kBoxBytes);
              tma_load_2d(xring + xs * kFXBox, &p.tmap_x, ks * 256 + hs * 128, m_tile * kRows, full_x + xs);
            }
            __syncwarp();
            filled_x |= 1u << xs;
            bits_x = (bits_x & ~(1u << xs)) | (xph << xs);
            ++xi;
            progressed = true;
          }
        }
        if (wi < my_st && __all_sync(0xFFFFFFFFu, mbar_test_wait(empty_w + wst, wph ^ 1u))) {
          const int ks = st0 + wi;
          const int nkk = min(4, KB / 4 - 4 * ks);
          uint8_t* b = wring + wst * kFWStage;
          uint8_t* sb = b + kFWTile;
          if (elect_one()) {
            mbar_arrive_expect_tx(full_w + wst, static_cast<uint32_t>(p.n_groups * (128 * 128 + 512 * nkk)));
            for (int h = 0; h < p.n_groups; ++h)                          // 128-row boxes
              tma_load_2d(b + h * 16384, &p.tmap_b, ks * 128, h * 128, full_w + wst);
            for (int h = 0; h < p.n_groups; ++h)
              bulk_load(sb + h * 2048, p.sfb + (static_cast<size_t>(h) * (KB / 4) + 4 * ks) * 512, 512u * nkk,
                        full_w + wst);
          }
          __syncwarp();
          filled_w |= 1u << wst;
          bits_w = (bits_w & ~(1u << wst)) | (wph << wst);
          if (++wst == kFStagesW) { wst = 0; wph ^= 1u; }
          ++wi;
          progressed = true;
        }
        if (!progressed) {
          __nanosleep(32);                               // leave the issue slots to the quantizer warps
          if ((++polls & 63) == 0 && (*abort_flag || globaltimer_ns() > deadline)) ok = false;
        }
      }
    } else {
      for (int s = 0; s < my_st && ok; ++s) {
        const int ks = st0 + s;
        // the stage's two x boxes (a box past D or T reads zeros)
        for (int hs = 0; hs < 2; ++hs, ++xi) {
          const int xs = xi % kFXSlots;
          const uint32_t xph = (xi / kFXSlots) & 1;
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty_x + xs, xph ^ 1u, deadline, abort_flag))) {
            ok = false;
            break;
          }
          if (elect_one()) {
            mbar_arrive_expect_tx(full_x + xs, kBoxBytes);
            tma_load_2d(xring + xs * kFXBox, &p.tmap_x, ks * 256 + hs * 128, m_tile * kRows, full_x + xs);
          }
          __syncwarp();
          filled_x |= 1u << xs;
          bits_x = (bits_x & ~(1u << xs)) | (xph << xs);
        }
        if (!ok) break;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty_w + wst, wph ^ 1u, deadline, abort_flag))) {
          ok = false;
          break;
        }
        const int nkk = min(4, KB / 4 - 4 * ks);
        uint8_t* b = wring + wst * kFWStage;
        uint8_t* sb = b + kFWTile;
        if (elect_one()) {
          mbar_arrive_expect_tx(full_w + wst, static_cast<uint32_t>(p.n_groups * (128 * 128 + 512 * nkk)));
          if (kNT == 2) {
            tma_load_2d(b, &p.tmap_b, ks * 128, 0, full_w + wst);      // 128 or 256 rows in one box
          } else {
            for (int h = 0; h < p.n_groups; ++h)                        // 128-row boxes
              tma_load_2d(b + h * 16384, &p.tmap_b, ks * 128, h * 128, full_w + wst);
          }
          for (int h = 0; h < p.n_groups; ++h)
            bulk_load(sb + h * 2048, p.sfb + (static_cast<size_t>(h) * (KB / 4) + 4 * ks) * 512, 512u * nkk,
                      full_w + wst);
        }
        __syncwarp();
        filled_w |= 1u << wst;
        bits_w = (bits_w & ~(1u << wst)) | (wph << wst);
        if (++wst == kFStagesW) { wst = 0; wph ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      report_timeout(p.status);
      *abort_flag = 1;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (!p.test_stall) {
      // kNT = 2: one MMA over the 128 or 256 experts; kNT = 3: experts
      // 0-255 (N = 256) and 256-383 (N = 128, accumulator columns 256 ..)
      const uint32_t idesc = idesc_mxf4nvf4(128, kNT == 2 ? 128 * p.n_groups : 256);
      const uint32_t idesc3 = idesc_mxf4nvf4(128, 128);
      int wst = 0;
      uint32_t wph = 0;
      bool ok = true;
      for (int s = 0; s < my_st; ++s) {
        const int slot = s & 1;
        const uint32_t aph = (s >> 1) & 1;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(q_done + slot, aph, deadline, abort_flag) &&
                                         mbar_wait(full_w + wst, wph, deadline, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int ks = st0 + s;
        const int nkk = min(4, KB / 4 - 4 * ks);
        const uint8_t* a = aring + slot * kFASlot;
        const uint8_t* b = wring + wst * kFWStage;
        const uint32_t sf_t = tmem + C::kScaleCol + slot * C::kScaleSlot;
        if (elect_one()) {
          // the stage's scale atoms into tensor memory (in order with the
          // MMAs on the tensor pipe): x at +4 kk, W group h at
          // +16 + 4 kNT kk + 4 h
          for (int kk = 0; kk < nkk; ++kk) {
            tc_copy_scales(sf_t + 4 * kk, desc_scale_tile(smem_u32(a + kFACodes + 512 * kk)));
            for (int h = 0; h < p.n_groups; ++h)
              tc_copy_scales(sf_t + 16 + 4 * kNT * kk + 4 * h,
                             desc_scale_tile(smem_u32(b + kFWTile + 2048 * h + 512 * kk)));
          }
          for (int kk = 0; kk < nkk; ++kk) {
            tc_mma_nvf4(tmem, desc_kmajor_sw128(smem_u32(a + 32 * kk)), desc_kmajor_sw128(smem_u32(b + 32 * kk)),
                        idesc, sf_t + 4 * kk, sf_t + 16 + 4 * kNT * kk, (s | kk) != 0);
            if (kNT == 3)
              tc_mma_nvf4(tmem + 256, desc_kmajor_sw128(smem_u32(a + 32 * kk)),
                          desc_kmajor_sw128(smem_u32(b + 256 * 128 + 32 * kk)), idesc3, sf_t + 4 * kk,
                          sf_t + 16 + 4 * kNT * kk + 8, (s | kk) != 0);
          }
          tc_commit(empty_w + wst);
          tc_commit(a_empty + slot);
        }
        __syncwarp();
        if (++wst == kFStagesW) { wst = 0; wph ^= 1u; }
      }
      if (ok && my_st > 0 && elect_one()) tc_commit(acc_full);
      __syncwarp();
      if (!ok && lane == 0) {
        report_timeout(p.status);
        *abort_flag = 1;
      }
    }
  } else {
    // ---------------------------------------------------------- quantizers
    rt.init(p.bias, p.N, p.k, p.raw, p.routed_scaling, lane);       // for the epilogue
    const float w_gsa = __ldg(p.w_gsa);                               // off the path after the barrier
    // quantizer warp q16 = warp - 2 takes the rows qw = q16 % 8 of box q16 / 8
    // of every stage
    const int q16 = warp - 2, qw = q16 & 7, qh = q16 >> 3;
    bool ok = true;
    int xi = 0;                                        // x boxes consumed so far
    // the grid barrier's generation, read before the max|x| pass so that the
    // barrier does not wait for it (after the grid-dependency wait the
    // previous call's bump is visible; this call bumps it only after every
    // CTA has arrived)
    const uint32_t gen = p.amax_sync && warp == 2 && lane == 0 ? ld_acquire_gpu(p.amax_sync + 4) : 0u;
    if (p.amax_sync) {
      // ---- in-kernel amax: max |x| over this CTA's boxes (the same
      // bit-pattern max as the amax kernel), then the grid-wide record
      uint32_t m = 0;
      for (int c = 0; c < n_chunks && ok; ++c) {
        const int cs = c % kFChunkSlots;
        const uint32_t cph = (c / kFChunkSlots) & 1;
        const bool okc = __all_sync(0xFFFFFFFFu, mbar_wait(full_c + cs, cph, deadline, abort_flag));
        ok = ok && okc;
        if (okc) {
          // warp q16 reads the box's 16-byte words q16 * 32 + lane + 512 i
          // (rows past T and columns past D are zeros)
          const uint8_t* cb = smem + cs * kFChunk;
#pragma unroll 4
          for (uint32_t o = (q16 * 32 + lane) * 16u; o < kBoxBytes; o += kFQThreads * 16u)
            m = max(m, absmax_bits16B<true>(ld_shared_v4(cb + o)));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_c + cs);
        if (!okc) break;
      }
      m = __reduce_max_sync(0xFFFFFFFFu, m);
      uint32_t* s_wmax = reinterpret_cast<uint32_t*>(s_fixq);     // the queue is not in use yet
      if (lane == 0) s_wmax[q16] = m;
      ok = bar_and(3, kFQThreads, ok);
      bool gok = true;
      if (warp == 2 && ok) {                           // ok is the same in every thread
        uint32_t cm = 0;
        for (int w = 0; w < kFQWarps; ++w) cm = max(cm, s_wmax[w]);
        uint32_t bits = 0;
        if (one_cluster) {
          // my maximum into slot `rank` of every CTA, then an arrival on its
          // mbarrier (release: the store is visible first) -- lane r serves
          // CTA r, so the S round trips overlap; then wait for all S
          uint32_t* s_cmax = reinterpret_cast<uint32_t*>(s_fixq) + 32;
          if (lane < p.S) {
            uint32_t slot, bar;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(slot) : "r"(smem_u32(s_cmax + rank)), "r"(lane));
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(bar) : "r"(smem_u32(amax_mbar)), "r"(lane));
            asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(slot), "r"(cm) : "memory");
            asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(bar) : "memory");
          }
          __syncwarp();
          if (lane == 0) {
            gok = false;
            for (uint32_t it = 0;; ++it) {
              uint32_t done;
              asm volatile("{\n\t.reg .pred q;\n\t"
                           "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 q, [%1], 0;\n\t"
                           "selp.u32 %0, 1, 0, q;\n\t}"
                           : "=r"(done) : "r"(smem_u32(amax_mbar)) : "memory");
              if (done) { gok = true; break; }
              if ((it & 63) == 63 && (*abort_flag || globaltimer_ns() > deadline)) break;
            }
            for (int r = 0; r < p.S; ++r) bits = max(bits, s_cmax[r]);
          }
        } else if (lane == 0) {
          gok = grid_amax(p.amax_sync, gen, cm, gridDim.x, bits, deadline, abort_flag);
        }
        if (lane == 0) {
          s_wmax[kFQWarps] = bits;
          if (!gok) {
            report_timeout(p.status);
            *abort_flag = 1;
          }
        }
      }
      ok = bar_and(3, kFQThreads, ok && gok);          // warp 2's outcome, for every warp
    }
    // the quantizer record: derived here from the grid's max (the amax
    // kernel's arithmetic; CTA 0 also stores it), or the amax kernel's
    QuantScale qs;
    float amax;
    if (p.amax_sync) {
      amax = __uint_as_float(reinterpret_cast<const uint32_t*>(s_fixq)[kFQWarps]);
      qs = make_quant_scale(amax);
      if (blockIdx.x == 0 && threadIdx.x == 64) {
        p.qrec[0] = qs.gsa;
        p.qrec[1] = qs.rgsa;
        p.qrec[2] = __int_as_float(qs.mode);
        p.qrec[3] = amax;
        *p.gsa_out = qs.gsa;
      }
      gscale = __fmul_rn(qs.gsa, w_gsa);
    } else {
      qs.gsa = __ldg(p.qrec);
      qs.rgsa = __ldg(p.qrec + 1);
      qs.mode = __float_as_int(__ldg(p.qrec + 2));
      amax = __ldg(p.qrec + 3);
      gscale = __fmul_rn(__ldg(p.x_gsa), w_gsa);
    }
    // bracketing quantizer (mode 1): the scale byte of every bf16 block max
    // within ~20 binades below amax, and the bracketing multipliers per byte
    const uint32_t amax_b16 = __float_as_uint(amax) >> 16;                  // bf16 bits of amax
    if (qs.mode == 1) {
      const float r6 = 0.16666667163372039794921875f;       // RN(1/6)
      const int qt = static_cast<int>(threadIdx.x) - 64;   // 0..511 over the quantizer warps
      static_assert(kFByteTab % kFQThreads == 0, "whole rounds of the table");
#pragma unroll
      for (int j = 0; j < kFByteTab / kFQThreads; ++j) {   // independent entries: their latencies overlap
        const int i = qt + kFQThreads * j;
        const int b16 = static_cast<int>(amax_b16) - i;
        const float mx = __uint_as_float(static_cast<uint32_t>(max(b16, 0)) << 16);
        s_byte[i] = static_cast<uint8_t>(e4m3_byte(div_rn_short(div_rn(mx, qs.gsa, qs.rgsa), 6.0f, r6)));
      }
      if (qt < 128) {
        const float c = __fmul_rn(qs.rgsa, s_scale[qt].y);   // RN(1/dec(b)), 0 for bytes 0 and 127
        s_cc[qt] = make_float2(__fmul_rn(c, 0.99999904632568359375f),     // 1 - 2^-20
                               __fmul_rn(c, 1.00000095367431640625f));    // 1 + 2^-20
      }
    }
    bar_and(2, kFQThreads, true);
    QuantTables tb;
    tb.qs = qs;
    tb.s_scale = s_scale;
    tb.s_cc = s_cc;
    tb.s_byte = s_byte;
    tb.amax_b16 = amax_b16;
    for (int s = 0; s < my_st; ++s) {
      const int slot = s & 1;
      const uint32_t aph = (s >> 1) & 1;
      // the slot is free once the MMAs that read it two stages ago completed
      // (no CTA-wide barrier: warps may run up to about a stage apart)
      if (!ok || !__all_sync(0xFFFFFFFFu, mbar_wait(a_empty + slot, aph ^ 1u, deadline, abort_flag))) {
        ok = false;
        break;
      }
      uint8_t* ac = aring + slot * kFASlot;
      uint8_t* asf = ac + kFACodes;
      {
        xi = 2 * s + qh;                               // box qh of the stage
        const int xs = xi % kFXSlots;
        const uint32_t xph = (xi / kFXSlots) & 1;
        const bool okx = __all_sync(0xFFFFFFFFu, mbar_wait(full_x + xs, xph, deadline, abort_flag));
        ok = ok && okx;
        if (okx) {
          quant_box<kRows>(xring + xs * kFXBox, ac, asf, qh, qw, lane, p.T - m_tile * kRows, tb,
                           s_fixq + q16 * kFFixQ);
        }
        // this warp has read its rows of the box
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_x + xs);
      }
      // the MMA reads the codes through the async proxy
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_done + slot);
    }
    if (!ok && lane == 0) {
      report_timeout(p.status);
      *abort_flag = 1;
    }
    // --------------------------------------------- wait for the accumulator
    if (my_st > 0) {
      acc_ok = bar_and(1, kFQThreads, mbar_wait(acc_full, 0, deadline, abort_flag));
      if (!acc_ok && threadIdx.x == 64) {
        report_timeout(p.status);
        *abort_flag = 1;
      }
    }
    tc_fence_after();
    // every x box and W tile has been read (the last MMA needed them all):
    // the rings stage the stores -- up to 256 experts two buffers per warp in
    // the W and x rings (contiguous), else one in the x ring
    static_assert(kNT == 3 || 16 * 2 * 4096 <= kFWRing + kFXRing, "two staging buffers per warp");
    static_assert(kFWRing % 1024 == 0, "the staging buffers are 1024-byte aligned (128-byte swizzle)");
    if constexpr (kNT == 2)
      store_partial_rows_tma<2>(&p.tmap_p, wring, tmem, warp, lane, m_tile * kRows, min(kRows, p.T - m_tile * kRows),
                                rank, p.n_groups, my_st > 0 && acc_ok, kFQWarps);
    else
      store_partial_rows_tma<1>(&p.tmap_p, xring, tmem, warp, lane, m_tile * kRows, min(kRows, p.T - m_tile * kRows),
                                rank, p.n_groups, my_st > 0 && acc_ok, kFQWarps);
  }

  // The S CTAs of this token tile form the cluster, or meet at the tile's
  // barrier in the workspace: after it every partial row of the tile is
  // visible to all of them.
  tc_fence_before();
  if (p.flat) {
    __syncthreads();
    if (threadIdx.x == 0 && p.S > 1 &&
        !tile_barrier(tile_count, static_cast<uint32_t>(p.S), deadline, abort_flag)) {
      report_timeout(p.status);
      *abort_flag = 1;
    }
    __syncthreads();
  } else {
    __syncwarp();
    cluster_sync_all();
  }
  tc_fence_after();

  // ------------------------------- router epilogue for this CTA's tokens
  // rank r finishes tokens [r * rows/S, (r+1) * rows/S) of the tile.  Router
  // warp rw (the quantizer warps) takes tokens rw, rw + 16, ..., one or two
  // per call (their latencies overlapping).
  const int per = kRows / p.S;
  if (warp >= 2) {
    const int rw = warp - 2;
    // with 8 or more partial planes (then at most 16 tokens per CTA: one per
    // router warp) and up to 256 experts the W and x rings (contiguous, idle
    // now) stage each warp's S partial rows, all copied at once (measured:
    // fewer planes are faster loaded directly): S KB per warp with a token,
    // rw < 128 / S; each warp's token slot is then in the A ring, else its
    // two slots are in the x ring (all idle now)
    constexpr int kSlot = RouteSlot<kNT>::kFloat4;
    const bool staged = kNT == 2 && p.S >= 8;
    float4* stage = staged ? reinterpret_cast<float4*>(wring) + rw * p.S * 64 : nullptr;
    static_assert(kNT == 3 || 128 * 1024 <= kFWRing + kFXRing, "epilogue staging fits the W and x rings");
    static_assert(kFQWarps * kSlot * 16 <= kFARing && 2 * kFQWarps * kSlot * 16 <= kFXRing,
                  "token slots fit the A ring (one per warp) and the x ring (two per warp)");
    float4* s_row = staged ? reinterpret_cast<float4*>(aring) + rw * kSlot
                           : reinterpret_cast<float4*>(xring) + rw * 2 * kSlot;
    const int64_t t0 = static_cast<int64_t>(m_tile) * kRows + static_cast<int64_t>(rank) * per;
    // as many token slots per call as the warp has tokens -- empty slots
    // would still be sorted
    const auto route_n = [&](auto nt) {
      constexpr int NT = decltype(nt)::value;
      for (int i = rw; i < per; i += kFQWarps * NT) {
        int64_t tt[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const int64_t t = t0 + i + kFQWarps * n;
          tt[n] = (i + kFQWarps * n < per && t < p.T) ? t : -1;
        }
        rt.template route<NT>(p.partials, static_cast<size_t>(p.T) * (128 * kNT), p.S, tt, gscale, s_row, lane,
                              p.out_ids, p.out_w, p.logits, stage);
      }
    };
    if (per <= kFQWarps) route_n(std::integral_constant<int, 1>());
    else route_n(std::integral_constant<int, 2>());
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort_flag && threadIdx.x == 0) {
    // After an abort, copies may still be landing in this CTA's shared
    // memory: wait (bounded) for the latest fill of every ring slot.
    const uint64_t drain = globaltimer_ns() + 1000000000ull;
    for (int s = 0; s < kFStagesW; ++s)
      while (((filled_w >> s) & 1u) && !mbar_try_wait(full_w + s, (bits_w >> s) & 1u))
        if (globaltimer_ns() > drain) break;
    for (int s = 0; s < kFXSlots; ++s)
      while (((filled_x >> s) & 1u) && !mbar_try_wait(full_x + s, (bits_x >> s) & 1u))
        if (globaltimer_ns() > drain) break;
    for (int s = 0; s < kFChunkSlots; ++s)
      while (((filled_c >> s) & 1u) && !mbar_try_wait(full_c + s, (bits_c >> s) & 1u))
        if (globaltimer_ns() > drain) break;
  }
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// bf16 activations [T, D]: boxes of box_rows rows x 128 elements, no swizzle,
// zeros outside.
bool encode_x(CUtensorMap* map, const uint16_t* ptr, int64_t T, int64_t D, uint32_t box_rows) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(ptr), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Per-device function attributes of the four instantiations (128- and
// 112-row tiles, heads of up to 256 and 384 experts): the dynamic shared
// memory and clusters of up to 16 CTAs (beyond the portable 8; the planner
// asks first).
static cudaError_t fused_prepare(int dev) {
  static bool done[kMaxDevices] = {};
  if (done[dev]) return cudaSuccess;
  struct Fn {
    void (*fn)(FusedParams);
    int smem;
  };
  const Fn fns[4] = {{fused_qgemm_kernel<128, 2>, FusedCfg<2>::kSmem}, {fused_qgemm_kernel<112, 2>, FusedCfg<2>::kSmem},
                     {fused_qgemm_kernel<128, 3>, FusedCfg<3>::kSmem}, {fused_qgemm_kernel<112, 3>, FusedCfg<3>::kSmem}};
  for (const Fn& f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, f.smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(f.fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  done[dev] = true;
  return cudaSuccess;
}

// How many CTAs of this kernel the device holds at once without clusters
// (cached per device; 0 on error).
int fused_block_capacity() {
  static int cap[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (cap[dev] > 0) return cap[dev];
  if (fused_prepare(dev) != cudaSuccess) return 0;
  int per_sm = 0;
  // the widest plan (one CTA per SM either way)
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_qgemm_kernel<128, 2>, kFThreads,
                                                    FusedCfg<2>::kSmem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cap[dev] = per_sm * device_sm_count();
  return cap[dev];
}

// How many clusters of S CTAs of this kernel the device can hold at once
// (cached per device and size; 0 when the size cannot be scheduled).
int fused_cluster_capacity(int S) {
  static int cap[kMaxDevices][5] = {};
  static bool known[kMaxDevices][5] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  const int slot = S == 1 ? 0 : S == 2 ? 1 : S == 4 ? 2 : S == 8 ? 3 : S == 16 ? 4 : -1;
  if (slot < 0) return 0;
  if (known[dev][slot]) return cap[dev][slot];
  if (fused_prepare(dev) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S);
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = FusedCfg<2>::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  // the widest plan (one CTA per SM either way)
  if (cudaOccupancyMaxActiveClusters(&n, fused_qgemm_kernel<128, 2>, &cfg) != cudaSuccess) n = 0;
  cudaGetLastError();
  cap[dev][slot] = n;
  known[dev][slot] = true;
  return n;
}

// per device: 0 unknown, 1 the runtime accepts the cooperative attribute with
// the router's others, -1 it refused it
static int g_fused_coop[kMaxDevices] = {};

nvr_status launch_fused_router(const uint16_t* x, float* qrec, float* x_gsa, uint32_t* amax_sync,
                               uint32_t* tile_sync, bool flat, int64_t T, int64_t D,
                               const uint8_t* W_codes, const uint8_t* W_sf, const float* w_gsa, int64_t N,
                               const float* bias, int k, float routed_scaling, bool raw, int32_t* out_ids,
                               float* out_w, float* logits, float* partials, uint32_t* status, int S,
                               int tile_rows, bool test_stall, bool cooperative, cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVR_ERR_CUDA;
  if (N > 384 || k > kMaxKmax || S < 1 || S > 16 || 128 % S) return NVR_ERR_UNSUPPORTED;
  if (tile_rows != 128 && tile_rows != 112) return NVR_ERR_UNSUPPORTED;
  if (amax_sync && !tile_sync) return NVR_ERR_INVALID_ARG;
  if (flat && (!amax_sync || (T + tile_rows - 1) / tile_rows > kMaxFlatTiles)) return NVR_ERR_UNSUPPORTED;
  if (static_cast<size_t>(S) * static_cast<size_t>((T + 127) / 128 * 128) > splitk_partial_rows(T))
    return NVR_ERR_UNSUPPORTED;
  const cudaError_t e = fused_prepare(dev);
  if (e != cudaSuccess) return cuda_status(e);
  FusedParams g;
  const int n_groups = static_cast<int>((N + 127) / 128);
  const int nt = N > 256 ? 3 : 2;
  if (!encode_x(&g.tmap_x, x, T, D, static_cast<uint32_t>(tile_rows))) return NVR_ERR_UNSUPPORTED;
  if (!encode_codes(&g.tmap_b, W_codes, N, D, nt == 2 ? 128u * n_groups : 128u)) return NVR_ERR_UNSUPPORTED;
  if (!encode_partial_rows(&g.tmap_p, partials, T, S, 128 * nt)) return NVR_ERR_UNSUPPORTED;
  g.qrec = qrec; g.sfb = W_sf; g.partials = partials;
  g.amax_sync = amax_sync; g.tile_sync = tile_sync; g.flat = flat ? 1 : 0; g.gsa_out = x_gsa;
  g.T = static_cast<int>(T); g.D = static_cast<int>(D); g.N = static_cast<int>(N); g.n_groups = n_groups; g.S = S;
  g.x_gsa = x_gsa; g.w_gsa = w_gsa; g.bias = raw ? nullptr : bias;
  g.k = k; g.raw = raw ? 1 : 0; g.routed_scaling = routed_scaling;
  g.out_ids = out_ids; g.out_w = out_w; g.logits = logits;
  g.status = status; g.test_stall = test_stall ? 1 : 0;
  cudaLaunchAttribute attr[3];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na++].val.programmaticStreamSerializationAllowed = 1;
  if (!flat) {                            // without clusters the tiles meet at tile_barrier
    attr[na].id = cudaLaunchAttributeClusterDimension;         // the S K-splits of a token tile
    attr[na].val.clusterDim.x = S;
    attr[na].val.clusterDim.y = 1;
    attr[na++].val.clusterDim.z = 1;
  }
  // With the in-kernel max|x| every CTA waits at a grid barrier (and without
  // clusters a tile's CTAs at a workspace barrier): a cooperative launch has
  // the runtime guarantee that the whole grid is resident at once, also next
  // to other kernels on other streams, instead of the host's occupancy
  // estimate alone.  Whether the runtime takes it together with programmatic
  // launch and clusters is found out once per device, on a call outside
  // stream capture (a launch the runtime refuses returns an error and runs
  // nothing); until then, and where it is refused, the launch is ordinary and
  // the barriers' bounded waits remain the safeguard.
  int* coop_ok = g_fused_coop;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  const bool capturing = cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone;
  const bool try_coop = cooperative && amax_sync && (coop_ok[dev] == 1 || (coop_ok[dev] == 0 && !capturing));
  if (try_coop) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na++].val.cooperative = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((T + tile_rows - 1) / tile_rows * S));
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = nt == 3 ? FusedCfg<3>::kSmem : FusedCfg<2>::kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  auto launch = [&]() {
    if (nt == 3)
      return tile_rows == 112 ? cudaLaunchKernelEx(&cfg, fused_qgemm_kernel<112, 3>, g)
                              : cudaLaunchKernelEx(&cfg, fused_qgemm_kernel<128, 3>, g);
    return tile_rows == 112 ? cudaLaunchKernelEx(&cfg, fused_qgemm_kernel<112, 2>, g)
                            : cudaLaunchKernelEx(&cfg, fused_qgemm_kernel<128, 2>, g);
  };
  cudaError_t e2 = launch();
  if (try_coop && coop_ok[dev] == 0) {
    if (e2 == cudaSuccess) {
      coop_ok[dev] = 1;
    } else {
      cudaGetLastError();                  // the refused launch ran nothing
      coop_ok[dev] = -1;
      cfg.numAttrs = na - 1;
      e2 = launch();
    }
  }
  return cuda_status(e2);
}

// 1 when the one-launch router's launches carry the cooperative attribute on
// the current device, -1 when the runtime refused it, 0 before the first
// one-launch call outside stream capture.
int fused_cooperative_state() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return g_fused_coop[dev];
}

}  // namespace nvr
