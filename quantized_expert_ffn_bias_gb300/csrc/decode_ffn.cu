// Expert FFN for small token counts (decode, MTP verify): HBM-bound dequant-GEMV.
//
// Each chosen expert's packed weights are streamed once per call for all the
// tokens routed to it (batch-union grouping, "25GB RAM runs 744B GLM-5.2" page
// (pwwt.cn), section 3.4) and dequantised as (code - zero_point) * scale
// ("Colibri walkthrough" page (discosf.com), section 3.4).
//
// Work unit = one warp: 16 rows of gate AND the same 16 rows of up (lanes
// 0-15 gate, 16-31 up; SwiGLU pairs lane r with lane r+16), or 32 rows of down
// (lane = row).  Every dot product is lane-local, so there is no cross-lane
// reduction, and all lanes read the same activation words (broadcast loads).
// Weights arrive by TMA in 128-byte column chunks of the unit's rows, 128B
// swizzled so that 8 lanes reading 8 rows hit 8 distinct bank groups.  Each
// warp runs its own mbarrier pipeline of kDecodeStages stages.
//
// Exact dequantisation in fp32: a 4-bit code c placed at mantissa bit 4p of
// 2^23 gives the float 2^23 + c*16^p; subtracting 2^23 + zp*16^p leaves
// (c - zp)*16^p exactly.  The activation was pre-multiplied by 16^-p (exact
// power of two), so the product equals (c - zp) * x.  Per 8 codes of a 32-bit
// word: 1 shift + 8 masks, 4 packed subtractions, 4 packed FMAs per token.
// int8 codes use byte positions (256^p) the same way.  Group partial sums are
// scaled by the fp16 group scale (int4) or, at the end, the row scale (int8).
#include "moe_internal.cuh"

namespace coli {

constexpr int kChunkRowsGU = kGateUpRows;                          // 16
constexpr int kStageBytesGU = 2 * kStageChunks * kGateUpRows * kChunk;  // gate + up
constexpr int kStageBytesD = kStageChunks * kDownRows * kChunk;
constexpr int kMaxTokPass = 8;
constexpr float kMagic = 8388608.0f;  // 2^23
constexpr uint32_t kMagicBits = 0x4B000000u;

struct Unit {
  int slot;      // expert slot (E = shared)
  int rb;        // row block
  int pbeg;      // first grouped pair row of the expert
  int cnt;       // number of tokens routed to the expert
  int N;         // rows of the streamed matrix
  int K;         // inputs of the streamed matrix
};

template <bool DOWN>
__device__ __forceinline__ bool get_unit(const FwdArgs& a, int u, int n_routed, Unit& out) {
  const int rows = DOWN ? kDownRows : kGateUpRows;
  const int per_routed = DOWN ? a.d / rows : a.F / rows;
  const int routed_units = n_routed * per_routed;
  int slot, rb;
  if (u < routed_units) {
    slot = a.unique[u / per_routed];
    rb = u % per_routed;
  } else {
    const int per_shared = DOWN ? a.d / rows : a.Fs / rows;
    if (!a.has_shared || u - routed_units >= per_shared) return false;
    slot = a.E;
    rb = u - routed_units;
  }
  out.slot = slot;
  out.rb = rb;
  out.pbeg = a.offsets[slot];
  out.cnt = a.offsets[slot + 1] - out.pbeg;
  const int Fe = slot == a.E ? a.Fs : a.F;
  out.N = DOWN ? a.d : Fe;
  out.K = DOWN ? Fe : a.d;
  return true;
}

__device__ __forceinline__ int n_units_of(const FwdArgs& a, int n_routed, bool down) {
  const int rows = down ? kDownRows : kGateUpRows;
  const int per_routed = down ? a.d / rows : a.F / rows;
  const int per_shared = a.has_shared ? (down ? a.d / rows : a.Fs / rows) : 0;
  return n_routed * per_routed + per_shared;
}

// Cursor over this warp's (unit, pass, k-block) sequence.
struct Cursor {
  int unit;      // global unit index (valid while < n_units)
  int pass;
  int kb;
  Unit u;
  int n_kb;
  int n_pass;
  bool valid;
};

template <int QT, bool DOWN>
__device__ __forceinline__ void cursor_load(const FwdArgs& a, int n_routed, int n_units, int unit, Cursor& c) {
  c.unit = unit;
  c.pass = 0;
  c.kb = 0;
  c.valid = unit < n_units && get_unit<DOWN>(a, unit, n_routed, c.u);
  if (c.valid) {
    const int row_bytes = QT == COLI_Q_INT4_G128 ? c.u.K / 2 : c.u.K;
    const int chunks = row_bytes / kChunk;
    c.n_kb = (chunks + kStageChunks - 1) / kStageChunks;
    c.n_pass = (c.u.cnt + kMaxTokPass - 1) / kMaxTokPass;
    if (c.n_pass == 0) c.valid = false;  // cannot happen for listed experts
  }
}

template <int QT, bool DOWN>
__device__ __forceinline__ void cursor_next(const FwdArgs& a, int n_routed, int n_units, int stride, Cursor& c) {
  if (++c.kb < c.n_kb) return;
  c.kb = 0;
  if (++c.pass < c.n_pass) return;
  cursor_load<QT, DOWN>(a, n_routed, n_units, c.unit + stride, c);
}

// Issue the TMA loads of one stage (lane 0 only).
template <int QT, bool DOWN>
__device__ __forceinline__ void issue_stage(const FwdArgs& a, const Cursor& c, uint8_t* stage, uint64_t* bar,
                                            uint64_t policy) {
  const int row_bytes = QT == COLI_Q_INT4_G128 ? c.u.K / 2 : c.u.K;
  const int chunks = row_bytes / kChunk;
  const int c0 = c.kb * kStageChunks;
  const int nc = min(kStageChunks, chunks - c0);
  const int rows = DOWN ? kDownRows : kGateUpRows;
  const int nmat = DOWN ? 1 : 2;
  mbar_arrive_expect_tx(bar, (uint32_t)(nmat * nc * rows * kChunk));
  for (int m = 0; m < nmat; ++m) {
    const CUtensorMap* map = a.maps + (size_t)c.u.slot * 3 + (DOWN ? 2 : m);
    for (int ci = 0; ci < nc; ++ci)
      tma_load_2d(stage + (m * kStageChunks + ci) * rows * kChunk, map, (c0 + ci) * kChunk, c.u.rb * rows, bar,
                  policy);
  }
}

// ------------------------------------------------------------------ per-stage math

// int4: accumulate one 16-byte piece (32 codes of one group) into acc2[t].
template <int NT>
__device__ __forceinline__ void piece_int4(uint4 w, const float* const* xrow, int k, const float2 (&cz)[4],
                                           float2 (&acc2)[kMaxTokPass]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t q = ws[i], v = q >> 12;
    const float2 f01 = make_float2(__uint_as_float((q & 0x0000000Fu) | kMagicBits),
                                   __uint_as_float((q & 0x000000F0u) | kMagicBits));
    const float2 f23 = make_float2(__uint_as_float((q & 0x00000F00u) | kMagicBits),
                                   __uint_as_float((q & 0x0000F000u) | kMagicBits));
    const float2 f45 = make_float2(__uint_as_float((q & 0x000F0000u) | kMagicBits),
                                   __uint_as_float((v & 0x00000F00u) | kMagicBits));
    const float2 f67 = make_float2(__uint_as_float((v & 0x0000F000u) | kMagicBits),
                                   __uint_as_float((v & 0x000F0000u) | kMagicBits));
    const float2 d01 = fsub2(f01, cz[0]), d23 = fsub2(f23, cz[1]), d45 = fsub2(f45, cz[2]),
                 d67 = fsub2(f67, cz[3]);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float4 xa = ldg_nc_f4(xrow[t] + k + 8 * i);
      const float4 xb = ldg_nc_f4(xrow[t] + k + 8 * i + 4);
      acc2[t] = ffma2(d01, make_float2(xa.x, xa.y), acc2[t]);
      acc2[t] = ffma2(d23, make_float2(xa.z, xa.w), acc2[t]);
      acc2[t] = ffma2(d45, make_float2(xb.x, xb.y), acc2[t]);
      acc2[t] = ffma2(d67, make_float2(xb.z, xb.w), acc2[t]);
    }
  }
}

// int8: one 16-byte piece = 16 codes.
template <int NT>
__device__ __forceinline__ void piece_int8(uint4 w, const float* const* xrow, int k, float2 cz,
                                           float2 (&acc2)[kMaxTokPass]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t q = ws[i], v = q >> 16;
    const float2 f01 = make_float2(__uint_as_float((q & 0x00FFu) | kMagicBits),
                                   __uint_as_float((q & 0xFF00u) | kMagicBits));
    const float2 f23 = make_float2(__uint_as_float((v & 0x00FFu) | kMagicBits),
                                   __uint_as_float((v & 0xFF00u) | kMagicBits));
    const float2 d01 = fsub2(f01, cz), d23 = fsub2(f23, cz);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float4 xa = ldg_nc_f4(xrow[t] + k + 4 * i);
      acc2[t] = ffma2(d01, make_float2(xa.x, xa.y), acc2[t]);
      acc2[t] = ffma2(d23, make_float2(xa.z, xa.w), acc2[t]);
    }
  }
}

__device__ __forceinline__ float f16_bits_to_float(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// One stage for one lane: its row `row` of matrix `mat`, chunk data at `buf`
// (rows x 128 B per chunk, swizzled).  acc[t] accumulates the dequantised dot.
template <int QT, int NT>
__device__ __forceinline__ void stage_compute(const DevMat& M, int row, int r_in_box, int rows_box, const uint8_t* buf,
                                              int kb, int nc, const float* const* xrow, float (&acc)[kMaxTokPass],
                                              float2 (&acc2)[kMaxTokPass], const float2& cz8) {
  const uint32_t base = smem_u32(buf);
  const int sw = r_in_box & 7;
  if (QT == COLI_Q_INT4_G128) {
    const int G = M.K / 128, ZB = (G + 1) / 2;
    const uint16_t* srow = static_cast<const uint16_t*>(M.s) + (size_t)row * G;
    const uint8_t* zrow = M.z + (size_t)row * ZB;
    for (int ci = 0; ci < nc; ++ci) {
      const int chunk = kb * kStageChunks + ci;
#pragma unroll
      for (int g2 = 0; g2 < 2; ++g2) {           // 256 codes per 128-byte chunk = 2 groups
        const int grp = chunk * 2 + g2;
        const float sc = f16_bits_to_float(__ldg(srow + grp));
        const uint32_t zb = __ldg(zrow + (grp >> 1));
        const float z = (float)((grp & 1) ? (zb >> 4) : (zb & 15u));
        const float2 cz[4] = {make_float2(kMagic + z, kMagic + 16.f * z),
                              make_float2(kMagic + 256.f * z, kMagic + 4096.f * z),
                              make_float2(kMagic + 65536.f * z, kMagic + 256.f * z),
                              make_float2(kMagic + 4096.f * z, kMagic + 65536.f * z)};
#pragma unroll
        for (int t = 0; t < NT; ++t) acc2[t] = make_float2(0.f, 0.f);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = g2 * 4 + jj;
          const uint4 w = lds128(base + ci * rows_box * kChunk + r_in_box * kChunk + ((j ^ sw) << 4));
          piece_int4<NT>(w, xrow, chunk * 256 + j * 32, cz, acc2);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t] = fmaf(sc, acc2[t].x + acc2[t].y, acc[t]);
      }
    }
  } else {
    for (int ci = 0; ci < nc; ++ci) {
      const int chunk = kb * kStageChunks + ci;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 w = lds128(base + ci * rows_box * kChunk + r_in_box * kChunk + ((j ^ sw) << 4));
        piece_int8<NT>(w, xrow, chunk * 128 + j * 16, cz8, acc2);
      }
    }
  }
}

template <int QT>
__device__ __forceinline__ float row_scale_int8(const DevMat& M, int row) {
  return __ldg(static_cast<const float*>(M.s) + row);
}

// Pre-scale of an activation that feeds the next dequant-GEMV at input index k.
template <int QT>
__device__ __forceinline__ float pos_scale_q(int k) {
  if (QT == COLI_Q_INT4_G128) {
    const int r = k & 7;
    const int p = r <= 4 ? r : r - 3;
    return __uint_as_float((uint32_t)(127 - 4 * p) << 23);
  }
  return (k & 1) ? (1.0f / 256.0f) : 1.0f;
}

// ------------------------------------------------------------------ one pass (NT tokens, all k-blocks)

template <int QT, bool DOWN, int NT>
__device__ __forceinline__ bool run_pass(const FwdArgs& a, int n_routed, int n_units, int stride, Cursor& cons,
                                         Cursor& prod, uint8_t* wbuf, uint64_t* bars, int& stage, uint32_t& phase,
                                         uint64_t policy) {
  const int lane = threadIdx.x & 31;
  const int rows_box = DOWN ? kDownRows : kGateUpRows;
  const int mat = DOWN ? 2 : (lane >> 4);
  const int r_in_box = DOWN ? lane : (lane & 15);
  const Unit u = cons.u;
  const int row = u.rb * rows_box + r_in_box;
  const DevMat M = a.experts[u.slot].m[mat];
  const int stage_bytes = DOWN ? kStageBytesD : kStageBytesGU;
  const int mat_off = DOWN ? 0 : mat * kStageChunks * rows_box * kChunk;
  const int row_bytes = QT == COLI_Q_INT4_G128 ? u.K / 2 : u.K;
  const int chunks = row_bytes / kChunk;

  // input rows of this pass
  const int p0 = u.pbeg + cons.pass * kMaxTokPass;
  const int ntok = min(kMaxTokPass, u.cnt - cons.pass * kMaxTokPass);
  const float* xrow[kMaxTokPass];
#pragma unroll
  for (int t = 0; t < kMaxTokPass; ++t) {
    const int tt = t < ntok ? t : 0;
    xrow[t] = DOWN ? a.h + (size_t)(p0 + tt) * a.Fmax : a.xs + (size_t)a.pair_token[p0 + tt] * a.d;
  }
  float acc[kMaxTokPass];
  float2 acc2[kMaxTokPass];
#pragma unroll
  for (int t = 0; t < kMaxTokPass; ++t) { acc[t] = 0.f; acc2[t] = make_float2(0.f, 0.f); }
  float2 cz8 = make_float2(0.f, 0.f);
  float s8 = 0.f;
  if (QT == COLI_Q_INT8_PC) {
    const float z = (float)__ldg(M.z + row);
    cz8 = make_float2(kMagic + z, kMagic + 256.f * z);
    s8 = row_scale_int8<QT>(M, row);
  }

  bool ok = true;
  for (int kb = 0; kb < cons.n_kb; ++kb) {
    uint64_t* bar = bars + stage;
    if (!mbar_wait(bar, phase)) { ok = false; break; }
    const int nc = min(kStageChunks, chunks - kb * kStageChunks);
    stage_compute<QT, NT>(M, row, r_in_box, rows_box, wbuf + stage * stage_bytes + mat_off, kb, nc, xrow, acc, acc2,
                          cz8);
    __syncwarp();
    if (prod.valid) {
      if (lane == 0) {
        fence_proxy_async_smem();
        issue_stage<QT, DOWN>(a, prod, wbuf + stage * stage_bytes, bar, policy);
      }
      cursor_next<QT, DOWN>(a, n_routed, n_units, stride, prod);
    }
    if (++stage == kDecodeStages) { stage = 0; phase ^= 1u; }
  }
  if (!ok) return false;

  if (QT == COLI_Q_INT8_PC) {
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = s8 * (acc2[t].x + acc2[t].y);
  }
  if (DOWN) {
#pragma unroll
    for (int t = 0; t < NT; ++t)
      if (t < ntok) a.y[(size_t)(p0 + t) * a.d + row] = acc[t];
  } else {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float upv = __shfl_down_sync(0xffffffffu, acc[t], 16);
      if (lane < 16 && t < ntok) {
        const float g = acc[t];
        const float hv = g / (1.0f + expf(-g)) * upv;
        a.h[(size_t)(p0 + t) * a.Fmax + row] = hv * pos_scale_q<QT>(row);
      }
    }
  }
  return true;
}

template <int QT, bool DOWN>
__global__ void __launch_bounds__(kDecodeWarps * 32, 1) decode_ffn_kernel(FwdArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t bars_all[kDecodeWarps][kDecodeStages];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stage_bytes = DOWN ? kStageBytesD : kStageBytesGU;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wbuf = smem + (size_t)warp * kDecodeStages * stage_bytes;
  uint64_t* bars = bars_all[warp];

  const int n_routed = a.n_unique[0];
  const int n_units = n_units_of(a, n_routed, DOWN);
  const int stride = gridDim.x * kDecodeWarps;
  const int first = blockIdx.x * kDecodeWarps + warp;
  if (first >= n_units) return;

  if (lane == 0) {
    for (int s = 0; s < kDecodeStages; ++s) mbar_init(bars + s, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t policy = l2_evict_first_policy();

  Cursor prod, cons;
  cursor_load<QT, DOWN>(a, n_routed, n_units, first, prod);
  cons = prod;
  for (int s = 0; s < kDecodeStages && prod.valid; ++s) {
    if (lane == 0) issue_stage<QT, DOWN>(a, prod, wbuf + s * stage_bytes, bars + s, policy);
    cursor_next<QT, DOWN>(a, n_routed, n_units, stride, prod);
  }
  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  while (cons.valid && ok) {
    const int ntok = min(kMaxTokPass, cons.u.cnt - cons.pass * kMaxTokPass);
    if (ntok <= 1) ok = run_pass<QT, DOWN, 1>(a, n_routed, n_units, stride, cons, prod, wbuf, bars, stage, phase, policy);
    else if (ntok <= 2) ok = run_pass<QT, DOWN, 2>(a, n_routed, n_units, stride, cons, prod, wbuf, bars, stage, phase, policy);
    else if (ntok <= 4) ok = run_pass<QT, DOWN, 4>(a, n_routed, n_units, stride, cons, prod, wbuf, bars, stage, phase, policy);
    else ok = run_pass<QT, DOWN, 8>(a, n_routed, n_units, stride, cons, prod, wbuf, bars, stage, phase, policy);
    // advance the consumer cursor to the next pass / unit
    cons.kb = cons.n_kb - 1;
    cursor_next<QT, DOWN>(a, n_routed, n_units, stride, cons);
  }
  if (!ok) {
    if (lane == 0) set_status(a.status, COLI_DEV_WAIT_TIMEOUT);
    // drain: wait (bounded) for every stage still in flight before the CTA's
    // shared memory can be released
    for (int s = 0; s < kDecodeStages; ++s) {
      const int st = (stage + s) % kDecodeStages;
      const uint32_t ph = phase ^ ((stage + s) >= kDecodeStages ? 1u : 0u);
      mbar_wait(bars + st, ph);
    }
  }
}

template <int QT, bool DOWN>
static cudaError_t launch_decode(const FwdArgs& a, cudaStream_t st, int num_sms) {
  const int stage_bytes = DOWN ? kStageBytesD : kStageBytesGU;
  const size_t smem = (size_t)kDecodeWarps * kDecodeStages * stage_bytes + 1024;
  auto kern = decode_ffn_kernel<QT, DOWN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms, kDecodeWarps * 32, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode_gateup(const FwdArgs& a, int, cudaStream_t st, int num_sms) {
  return a.qtype == COLI_Q_INT4_G128 ? launch_decode<COLI_Q_INT4_G128, false>(a, st, num_sms)
                                     : launch_decode<COLI_Q_INT8_PC, false>(a, st, num_sms);
}

cudaError_t launch_decode_down(const FwdArgs& a, int, cudaStream_t st, int num_sms) {
  return a.qtype == COLI_Q_INT4_G128 ? launch_decode<COLI_Q_INT4_G128, true>(a, st, num_sms)
                                     : launch_decode<COLI_Q_INT8_PC, true>(a, st, num_sms);
}

}  // namespace coli
