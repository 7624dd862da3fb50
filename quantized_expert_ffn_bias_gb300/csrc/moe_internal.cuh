// Internal definitions shared by the kernels and the C-ABI layer of the
// quantized sparse MoE layer library.  sm_103a only.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/colibri_moe.h"

namespace coli {

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kDecodeMaxT = 8;          // tokens per forward served by the dequant-GEMV kernels
constexpr float kNearTie = 1e-5f;       // k-th minus (k+1)-th selection score below this = near-tie
constexpr int kRouterKSplit = 4;        // K-splits of the router logits (partial sums summed in order)

// ---------------------------------------------------------------- device tables

// One expert's three packed matrices (device pointers) and sizes.
struct DevMat {
  const uint8_t* q;
  const void* s;
  const uint8_t* z;
  int N, K;
};
struct DevExpert {
  DevMat m[3];  // 0 gate [F][d], 1 up [F][d], 2 down [d][F]
  int F;
  int pad_;
};

// TMA boxes of the decode (dequant-GEMV) kernels: 256-byte column slices of
// 8 rows (gate, up) or 16 rows (down), unswizzled.
constexpr int kTmaBoxBytes = 256;
constexpr int kGateUpBoxRows = 8;
constexpr int kDownBoxRows = 16;
#ifndef COLI_DECODE_STAGES
#define COLI_DECODE_STAGES 3
#endif
#ifndef COLI_DECODE_WARPS
#define COLI_DECODE_WARPS 8
#endif
constexpr int kDecodeStages = COLI_DECODE_STAGES;   // pipeline depth per warp
constexpr int kDecodeWarps = COLI_DECODE_WARPS;     // warps per CTA, each with its own pipeline
constexpr int kXsumBlock = 16;           // activation block sums are kept per 16 inputs

// ---------------------------------------------------------------- workspace layout

// Offsets (bytes) into the caller's workspace; computed by the plan.
struct WsLayout {
  size_t status;       // int32[16]: [0] status bits, [1] router last-CTA counter
  size_t topk_idx;     // int32 [T_max][k]
  size_t topk_w;       // float [T_max][k]
  size_t near_tie;     // int32 [T_max]
  size_t offsets;      // int32 [E+2]; offsets[E]..[E+1] = shared rows
  size_t pair_token;   // int32 [P_max + T_max]
  size_t pair_slot;    // int32 [P_max]
  size_t pair_of;      // int32 [P_max]
  size_t unique;       // int32 [E+1]
  size_t utab;         // int4 [E+1]: (slot, first pair row, pairs, 0) per expert with tokens, most pairs first, then the shared expert; decode only
  size_t n_unique;     // int32 [4]
  size_t logits;       // float [kRouterKSplit][T_max][E]
  size_t xs;           // float [T_max][d]  (dequant-GEMV input, pre-scaled)
  size_t xsum;         // float [T_max][d / kXsumBlock]  (unscaled block sums of x)
  size_t xq;           // uint32 [T_max][d / 2]  16-bit fixed-point x as int8 hi / uint8 lo bytes (int4 decode)
  size_t xqs;          // int2 [T_max][d / kXqBlock]  (block scale bits, sum of the fixed-point values)
  size_t h;            // float [P_max + T_max][Fmax]  (pre-scaled SwiGLU output)
  size_t hsum;         // float [P_max + T_max][Fmax / 8]  (unscaled sums of h over 8 rows)
  size_t hq;           // uint32 [P_max + T_max][Fmax / 2]  h in the fixed-point layout of xq (int4 decode)
  size_t hqs;          // int2 [P_max + T_max][Fmax / kXqBlock]
  size_t y;            // float [P_max + T_max][d]
  // tensor-core path (T_max > kDecodeMaxT only; 0 otherwise)
  size_t xh;           // fp16 [P_max + T_max][d]  activations in grouped order
  size_t chunks;       // chunk table (16 B each)
  size_t gu_tiles;     // gate/up tile table (16 B each)
  size_t dn_tiles;     // down tile table (16 B each)
  size_t pf_counts;    // int32[4]: chunks, gate/up tiles, down tiles
  size_t wsplit;       // bf16 [3][E][d] router weights in three parts (tensor-core router; 0 if unused)
  size_t total;
};

// Everything a kernel needs to know about one forward call.
struct FwdArgs {
  const DevExpert* experts;   // [n_slots + 1] expert descriptors by storage slot (the last one: shared)
  const CUtensorMap* maps;    // [(n_slots+1)*3] dequant-GEMV maps, then [(n_slots+1)*3] tensor-core maps
  const int32_t* slot_of;     // [E+1] storage slot of each expert id (E = shared); NULL: slot = expert id
  int T, d, F, Fs, E, k, qtype, xtype, has_shared;
  float rho;
  int Fmax;                   // row stride of h
  const void* x;
  const float* router_w;
  const float* bias;
  const float* residual;
  float* out;
  int32_t* status;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* near_tie;
  int32_t* offsets;
  int32_t* pair_token;
  int32_t* pair_slot;
  int32_t* pair_of;
  int32_t* unique;
  int4* utab;
  int32_t* n_unique;
  float* logits;
  float* xs;
  float* xsum;
  uint32_t* xq;
  int2* xqs;                  // per block of kXqBlock inputs: (block scale bits, sum of the fixed-point values)
  float* h;
  float* hsum;
  uint32_t* hq;
  int2* hqs;
  float* y;
  unsigned long long wait_ns; // limit of every pipeline wait (kWaitLimitNs unless a test shortens it)
  int inject;                 // COLI_INJECT_* bits of a failure-path test, 0 in normal use
  int idot;                   // 1: integer-dot inputs (int8 codes per block of 32, power-of-two scale)
};

// ---------------------------------------------------------------- launchers (one .cu file each)

cudaError_t launch_route_decode(const FwdArgs& a, cudaStream_t st);
cudaError_t launch_router_logits(const FwdArgs& a, cudaStream_t st);
// Router logits on the tensor cores (bf16 x, T >= kRouterTcMinT, d / kRouterKSplit a multiple of 64):
// the fp32 router weights split into three bf16 parts in the workspace, then one grouped MMA pass.
constexpr int kRouterTcMinT = 128;
bool router_tc_applies(const FwdArgs& a);
cudaError_t launch_router_split(const FwdArgs& a, void* wsplit, cudaStream_t st);
cudaError_t launch_router_tc(const FwdArgs& a, const void* wsplit, PFN_cuTensorMapEncodeTiled_v12000 encode,
                             cudaStream_t st);
cudaError_t launch_router_topk(const FwdArgs& a, cudaStream_t st);
cudaError_t launch_permute(const FwdArgs& a, cudaStream_t st);
cudaError_t launch_quantize_h(const FwdArgs& a, cudaStream_t st);
// The down kernels' input as floats (colibri_moe_debug_hidden).  mode: 0 decode
// 16-bit fixed point (int4), 1 decode pre-scaled fp32 (int8), 2 decode int8
// codes in unpack order (int4, integer-dot), 3 the same in natural order
// (int8, integer-dot), 4 prefill fp16 (column-permuted when perm).
struct HiddenView {
  int mode, perm, qtype, rows, P, F, Fs, Fmax;
  const float* h;
  const uint8_t* hq;
  const int2* hqs;
  const __half* hh;
  float* out;
};
cudaError_t launch_debug_hidden(const HiddenView& v, cudaStream_t st);
cudaError_t launch_decode_gateup(const FwdArgs& a, int max_tok_per_expert, cudaStream_t st, int num_sms);
cudaError_t launch_decode_down(const FwdArgs& a, int max_tok_per_expert, cudaStream_t st, int num_sms);
cudaError_t launch_combine(const FwdArgs& a, cudaStream_t st);
cudaError_t launch_rmsnorm_bf16(const float* h, int T, int d, float eps, uint16_t* out, cudaStream_t st);
cudaError_t launch_gather_x(const FwdArgs& a, __half* xh, int rows, cudaStream_t st);
cudaError_t launch_plan_tiles(const FwdArgs& a, void* chunks, void* gu_tiles, void* dn_tiles, int32_t* counts,
                              cudaStream_t st);
cudaError_t launch_prefill_gateup(const FwdArgs& a, const void* chunks, const void* tiles, const int32_t* n_tiles,
                                  const CUtensorMap* wmaps, const CUtensorMap& xmap, __half* hout, cudaStream_t st,
                                  int num_sms);
cudaError_t launch_prefill_down(const FwdArgs& a, const void* chunks, const void* tiles, const int32_t* n_tiles,
                                const CUtensorMap* wmaps, const CUtensorMap& hmap, float* yout, cudaStream_t st,
                                int num_sms);
// One call of the sparse-attention key selection (indexer.cu): T query tokens at positions
// pos0 .. pos0 + T - 1, each with 64 heads of 128 bf16 values (q [T][64][128]) and 64 fp32
// head weights (w [T][64]); L bf16 keys [L][128]; scores [T][L] fp32 and the selection
// out [T][topk] int32 (ascending keys, -1 padded) in caller memory.
struct IndexerCall {
  int T, L, pos0, topk;
  const void* q;
  const float* w;
  const void* keys;
  float* scores;         // [T][L]
  int32_t* out;
  int32_t* status;
  unsigned long long wait_ns;
  PFN_cuTensorMapEncodeTiled_v12000 encode;
  int steps;             // 1: scores, 2: selection from the scores, 3: both
};
cudaError_t launch_indexer(const IndexerCall& c, cudaStream_t st, int num_sms);
cudaError_t launch_indexer_scores(const IndexerCall& c, cudaStream_t st, int num_sms);

// int4 decode activations in 16-bit fixed point per block of kXqBlock inputs:
// x ~= sx * q with sx a power of two (|q| < 2^15), q = 256 * hi + lo with hi a
// signed and lo an unsigned byte.  Within a block, 64 bytes: 8 words of hi then
// 8 words of lo; word 2w (2w+1) holds the bytes of inputs 8w+0,2,4,6 (8w+1,3,5,7),
// the order in which the low (high) nibbles of a 32-bit word of codes unpack.
constexpr int kXqBlock = 32;

constexpr int kPrefillRows = 128;   // weight rows per tensor-core tile (box height of the raw-code maps)
#ifndef COLI_PREFILL_CHUNK
#define COLI_PREFILL_CHUNK 128
#endif
constexpr int kPrefillChunk = COLI_PREFILL_CHUNK;  // tokens per chunk (largest MMA N): 64 or 128
// Activation rows per TMA box of the tensor-core kernels (a chunk of n tokens loads
// ceil(n / kPrefillBBox) boxes per 64-column atom).  Each TMA instruction costs the
// single producer thread far more than the rows it moves: 64-row boxes measured
// faster than 16-row boxes, which load only the rows the MMAs read.
#ifndef COLI_PREFILL_BBOX
#define COLI_PREFILL_BBOX 64
#endif
constexpr int kPrefillBBox = COLI_PREFILL_BBOX;
static_assert(kPrefillBBox % 16 == 0 && kPrefillBBox <= kPrefillChunk && kPrefillBBox <= 256, "activation box");

// K extent of one pipeline stage of the tensor-core path (128: one int4 group
// per stage; gate/up stages carry both matrices).  The raw-code TMA box of a
// matrix is one stage wide.
__host__ __device__ constexpr int prefill_stage_k(bool gate_up) { return gate_up ? 128 : 128; }
__host__ __device__ constexpr int prefill_raw_row_bytes(int qtype, bool gate_up) {
  return qtype == COLI_Q_INT4_G128 ? prefill_stage_k(gate_up) / 2 : prefill_stage_k(gate_up);
}

// ---------------------------------------------------------------- device helpers

#ifdef __CUDACC__

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // default: give up a pipeline wait after ~1 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of an mbarrier; false after limit_ns nanoseconds (the
// caller then records COLI_DEV_WAIT_TIMEOUT and stops using the pipeline).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && globaltimer() - t0 > limit_ns) return false;
  }
}

// Non-blocking probe of an mbarrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Spinning wait for the thread that issues tensor-core instructions: the MMA
// stream stalls while that thread is busy, and a test_wait on a completed
// phase returns several times faster than a try_wait.  Bounded like mbar_wait.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && globaltimer() - t0 > limit_ns) return false;
  }
}

// One warp converts a block of kXqBlock = 32 values (lane i holds value i) to
// the fixed-point layout described at kXqBlock: 64 bytes at dst and
// (sx bits, sum of q) at *qs.  sx = 2^(floor(log2 max|v|) - 14).
__device__ __forceinline__ void warp_quantize_block32(float v, uint8_t* dst, int2* qs) {
  const int lane = threadIdx.x & 31;
  float m = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  int e = (int)((__float_as_uint(m) >> 23) & 255u) - 127;
  e = e < -100 ? -100 : e;                       // tiny blocks
  const float sx = __uint_as_float((uint32_t)(e - 14 + 127) << 23);
  const float inv = __uint_as_float((uint32_t)(14 - e + 127) << 23);
  int q = __float2int_rn(v * inv);
  q = q > 32767 ? 32767 : (q < -32767 ? -32767 : q);
  int sum = q;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const int j = lane & 7, wd = (lane >> 3) * 2 + (j & 1);
  dst[wd * 4 + (j >> 1)] = (uint8_t)((q >> 8) & 255);          // hi (two's complement byte)
  dst[32 + wd * 4 + (j >> 1)] = (uint8_t)(q & 255);             // lo
  if (lane == 0) *qs = make_int2(__float_as_int(sx), sum);
}

// Integer-dot (IDOT) inputs: one warp quantises one block of 32 values (lane i
// holds value i) to int8 codes q = rint(v / 2^(e-6)), clamped to [-127, 127],
// with e = floor(log2(max |v|)) read from the exponent bits of the block's
// largest magnitude (at least -100, so that 2^(e-6) and 2^(6-e) are normal
// floats).  v * 2^(6-e) is exact, so the codes do not depend on the
// arithmetic's precision.  NATURAL: code i at byte i (int8 weights); else in
// the nibble-unpack order of the int4 kernels (the hi-byte positions of
// warp_quantize_block32).  qs = (bits of 2^(e-6), sum of the codes).
template <bool NATURAL>
__device__ __forceinline__ void warp_quantize_block32_i8(float v, uint8_t* dst, int2* qs) {
  const int lane = threadIdx.x & 31;
  float m = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  int e = (int)((__float_as_uint(m) >> 23) & 255u) - 127;
  e = e < -100 ? -100 : e;
  const float sx = __uint_as_float((uint32_t)(e - 6 + 127) << 23);
  const float inv = __uint_as_float((uint32_t)(6 - e + 127) << 23);
  int q = __float2int_rn(v * inv);
  q = q > 127 ? 127 : (q < -127 ? -127 : q);
  int sum = q;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (NATURAL) {
    dst[lane] = (uint8_t)(q & 255);
  } else {
    const int j = lane & 7, wd = (lane >> 3) * 2 + (j & 1);
    dst[wd * 4 + (j >> 1)] = (uint8_t)(q & 255);
  }
  if (lane == 0) *qs = make_int2(__float_as_int(sx), sum);
}

// The IDOT value q * 2^(e-6) of v, given the block's largest magnitude m
// (prefill: the tensor-core operands carry these values in fp16).
__device__ __forceinline__ float idot_value(float v, float m) {
  int e = (int)((__float_as_uint(m) >> 23) & 255u) - 127;
  e = e < -100 ? -100 : e;
  const float sx = __uint_as_float((uint32_t)(e - 6 + 127) << 23);
  const float inv = __uint_as_float((uint32_t)(6 - e + 127) << 23);
  int q = __float2int_rn(v * inv);
  q = q > 127 ? 127 : (q < -127 ? -127 : q);
  return (float)q * sx;
}

// Programmatic dependent launch: a kernel launched with launch_pdl may start
// while the previous kernel on the stream is still running; griddep_wait()
// blocks until that kernel has completed and its writes are visible, and
// griddep_launch_dependents() lets the next kernel start its own prologue.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Make generic-proxy shared-memory accesses ordered before later async-proxy
// (TMA / tensor core) accesses of this thread.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2D tiled TMA load into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ------------------------------------------------------------------ tcgen05 and TMA helpers

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// atoms 1024 bytes apart (the layout a 128-byte-swizzled TMA box produces).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                       // leading byte offset (unused: K extent within one atom)
  d |= (uint64_t)(1024 >> 4) << 32;             // stride byte offset: next 8 rows
  d |= (uint64_t)1 << 46;                       // descriptor version
  d |= (uint64_t)2 << 61;                       // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: fp16 A and B (K-major), fp32 accumulate.
__device__ __forceinline__ uint32_t umma_idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The same with bf16 A and B.
__device__ __forceinline__ uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// One MMA with both operands in shared memory (descriptors a, b); acc = 0 overwrites the accumulators.
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive TMEM columns of this warp's 32 lanes -> registers (issue only)
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// registers -> 16 consecutive TMEM columns of this warp's 32 lanes
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2D TMA load without cache hint.
__device__ __forceinline__ void tma_load_2d_nohint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Prefetch a 2D box of a tensor into L2 (no shared-memory destination).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// L2 policy for data read exactly once per call (streamed expert weights).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- packed fp32x2 arithmetic (two lanes per instruction)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ float4 ldg_nc_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void set_status(int32_t* status, int32_t bits) { atomicOr(status, bits); }

// Block-wide exclusive prefix sum of one int per thread (blockDim.x a multiple
// of 32, <= 1024).  *total receives the block sum.  Contains __syncthreads().
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nw ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < nw) warp_tot[lane] = wi - w;  // exclusive warp offsets
    if (lane == nw - 1) *total = wi;
  }
  __syncthreads();
  const int r = warp_tot[warp] + inc - v;
  __syncthreads();
  return r;
}

// Activation pre-scale for the dequant-GEMV at input index k: the kernels form
// code * 16^p (int4, p = 0,1,2,3,4,2,3,4 for k mod 8) or code * 256^(k mod 2)
// (int8) exactly, so the activation carries the inverse power of two (exact).
__device__ __forceinline__ float act_prescale(int qtype, int k) {
  if (qtype == COLI_Q_INT4_G128) {
    const int r = k & 7;
    const int p = r <= 4 ? r : r - 3;
    return __uint_as_float((uint32_t)(127 - 4 * p) << 23);
  }
  return (k & 1) ? (1.0f / 256.0f) : 1.0f;
}

#endif  // __CUDACC__

}  // namespace coli
