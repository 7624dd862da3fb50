// Expert FFN for small token counts (decode, MTP verify): HBM-bound dequant-GEMV.
//
// Each chosen expert's packed weights are streamed once per call for all the
// tokens routed to it (batch-union grouping, "25GB RAM runs 744B GLM-5.2" page
// (pwwt.cn), section 3.4) and dequantised as (code - zero_point) * scale
// ("Colibri walkthrough" page (discosf.com), section 3.4).
//
// Work unit = one warp and 16 matrix rows: 8 rows of gate with the same 8
// rows of up (SwiGLU needs both), or 16 rows of down.  A pipeline stage holds
// 512 bytes of each of the 16 rows (TMA, two 256-byte boxes per row block);
// lane l owns bytes [16l, 16l+16) of every row of the stage, i.e. 32 int4 or
// 16 int8 codes.  The lane's activations for those codes are loaded once per
// stage and reused for all 16 rows, and the 16 rows give 16 independent
// accumulation chains.  After the last stage a butterfly reduction across the
// 32 lanes leaves row r in lanes 2r and 2r+1.  Each warp runs its own
// kDecodeStages-deep mbarrier pipeline.
//
// Exact dequantisation in fp32: a code c placed at mantissa bit 4p (int4) or
// 8p (int8) of the float 2^23 gives 2^23 + c*16^p; subtracting 2^23 leaves
// c*16^p exactly, and the activation was pre-multiplied by 16^-p (an exact
// power of two), so the product is c*x.  The zero-point is applied once per
// (row, 32-code slice): sum((c - z) x) = sum(c x) - z sum(x).  Group sums are
// scaled by the fp16 group scale (int4) or, at the end, by the row scale (int8).
#include "moe_internal.cuh"

namespace coli {

constexpr int kUnitRows = 16;              // rows per warp unit (gate/up: 8 + 8)
constexpr int kRowBytesPerStage = 512;     // bytes of each row per stage
constexpr int kBoxBytes = kTmaBoxBytes;    // TMA box inner extent
constexpr int kStageBytes = kUnitRows * kRowBytesPerStage;  // 8 KB
constexpr float kMagic = 8388608.0f;       // 2^23
constexpr uint32_t kMagicBits = 0x4B000000u;

struct Unit {
  int slot;   // expert slot (E = shared)
  int rb;     // row block (8 rows of gate/up, or 16 rows of down)
  int pbeg;   // first grouped pair row of the expert
  int cnt;    // tokens routed to the expert
  int K;      // inputs of the streamed matrix
};

static_assert(kGateUpBoxRows == kUnitRows / 2 && kDownBoxRows == kUnitRows, "TMA boxes must match the unit rows");

template <bool DOWN>
__device__ __forceinline__ int rows_per_unit() { return DOWN ? kUnitRows : kUnitRows / 2; }

template <bool DOWN>
__device__ __forceinline__ bool get_unit(const FwdArgs& a, int u, int n_routed, Unit& out) {
  const int rows = rows_per_unit<DOWN>();
  const int per_routed = (DOWN ? a.d : a.F) / rows;
  const int routed_units = n_routed * per_routed;
  int slot, rb;
  if (u < routed_units) {
    slot = a.unique[u / per_routed];
    rb = u % per_routed;
  } else {
    const int per_shared = (DOWN ? a.d : a.Fs) / rows;
    if (!a.has_shared || u - routed_units >= per_shared) return false;
    slot = a.E;
    rb = u - routed_units;
  }
  out.slot = slot;
  out.rb = rb;
  out.pbeg = a.offsets[slot];
  out.cnt = a.offsets[slot + 1] - out.pbeg;
  const int Fe = slot == a.E ? a.Fs : a.F;
  out.K = DOWN ? Fe : a.d;
  return true;
}

template <bool DOWN>
__device__ __forceinline__ int n_units_of(const FwdArgs& a, int n_routed) {
  const int rows = rows_per_unit<DOWN>();
  const int per_routed = (DOWN ? a.d : a.F) / rows;
  const int per_shared = a.has_shared ? (DOWN ? a.d : a.Fs) / rows : 0;
  return n_routed * per_routed + per_shared;
}

template <int QT>
__device__ __forceinline__ int row_bytes_of(int K) { return QT == COLI_Q_INT4_G128 ? K / 2 : K; }

// Cursor over this warp's (unit, pass, stage) sequence.
struct Cursor {
  int unit;
  int pass;
  int kb;
  int n_kb;
  int n_pass;
  bool valid;
  Unit u;
};

template <int QT, bool DOWN, int NTMAX>
__device__ __forceinline__ void cursor_load(const FwdArgs& a, int n_routed, int n_units, int unit, Cursor& c) {
  c.unit = unit;
  c.pass = 0;
  c.kb = 0;
  c.valid = unit < n_units && get_unit<DOWN>(a, unit, n_routed, c.u);
  if (c.valid) {
    c.n_kb = (row_bytes_of<QT>(c.u.K) + kRowBytesPerStage - 1) / kRowBytesPerStage;
    c.n_pass = (c.u.cnt + NTMAX - 1) / NTMAX;
    c.valid = c.n_pass > 0;
  }
}

template <int QT, bool DOWN, int NTMAX>
__device__ __forceinline__ void cursor_next(const FwdArgs& a, int n_routed, int n_units, int stride, Cursor& c) {
  if (++c.kb < c.n_kb) return;
  c.kb = 0;
  if (++c.pass < c.n_pass) return;
  cursor_load<QT, DOWN, NTMAX>(a, n_routed, n_units, c.unit + stride, c);
}

// TMA loads of one stage (lane 0): for each matrix, the unit's rows x up to
// two 256-byte boxes.  Shared layout: [matrix][box half][rows][256 B].
template <int QT, bool DOWN>
__device__ __forceinline__ void issue_stage(const FwdArgs& a, const Cursor& c, uint8_t* stage, uint64_t* bar,
                                            uint64_t policy) {
  const int rb_bytes = row_bytes_of<QT>(c.u.K);
  const int x0 = c.kb * kRowBytesPerStage;
  const int nbox = x0 + kBoxBytes < rb_bytes ? 2 : 1;
  const int rows = rows_per_unit<DOWN>();
  const int nmat = DOWN ? 1 : 2;
  mbar_arrive_expect_tx(bar, (uint32_t)(nmat * nbox * rows * kBoxBytes));
  for (int m = 0; m < nmat; ++m) {
    const CUtensorMap* map = a.maps + (size_t)c.u.slot * 3 + (DOWN ? 2 : m);
    for (int h = 0; h < nbox; ++h)
      tma_load_2d(stage + (m * 2 + h) * rows * kBoxBytes, map, x0 + h * kBoxBytes, c.u.rb * rows, bar, policy);
  }
}

__device__ __forceinline__ float f16_bits_to_float(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// position scales 16^p of the int4 codes of one 32-bit word (p = 0,1,2,3,4,2,3,4)
__device__ __forceinline__ float int4_pos_scale(int i) {
  const int r = i & 7;
  const int p = r <= 4 ? r : r - 3;
  return __uint_as_float((uint32_t)(127 + 4 * p) << 23);
}

// sum over one 32-bit word of int4 codes of c * x'  (x' pre-scaled), packed
__device__ __forceinline__ float2 dot_word_int4(uint32_t q, const float* xp, float2 acc) {
  const uint32_t v = q >> 12;
  const float2 M2 = make_float2(kMagic, kMagic);
  const float2 d01 = fsub2(make_float2(__uint_as_float((q & 0x0000000Fu) | kMagicBits),
                                       __uint_as_float((q & 0x000000F0u) | kMagicBits)), M2);
  const float2 d23 = fsub2(make_float2(__uint_as_float((q & 0x00000F00u) | kMagicBits),
                                       __uint_as_float((q & 0x0000F000u) | kMagicBits)), M2);
  const float2 d45 = fsub2(make_float2(__uint_as_float((q & 0x000F0000u) | kMagicBits),
                                       __uint_as_float((v & 0x00000F00u) | kMagicBits)), M2);
  const float2 d67 = fsub2(make_float2(__uint_as_float((v & 0x0000F000u) | kMagicBits),
                                       __uint_as_float((v & 0x000F0000u) | kMagicBits)), M2);
  acc = ffma2(d01, make_float2(xp[0], xp[1]), acc);
  acc = ffma2(d23, make_float2(xp[2], xp[3]), acc);
  acc = ffma2(d45, make_float2(xp[4], xp[5]), acc);
  acc = ffma2(d67, make_float2(xp[6], xp[7]), acc);
  return acc;
}

__device__ __forceinline__ float2 dot_word_int8(uint32_t q, const float* xp, float2 acc) {
  const uint32_t v = q >> 16;
  const float2 M2 = make_float2(kMagic, kMagic);
  const float2 d01 = fsub2(make_float2(__uint_as_float((q & 0x00FFu) | kMagicBits),
                                       __uint_as_float((q & 0xFF00u) | kMagicBits)), M2);
  const float2 d23 = fsub2(make_float2(__uint_as_float((v & 0x00FFu) | kMagicBits),
                                       __uint_as_float((v & 0xFF00u) | kMagicBits)), M2);
  acc = ffma2(d01, make_float2(xp[0], xp[1]), acc);
  acc = ffma2(d23, make_float2(xp[2], xp[3]), acc);
  return acc;
}

// Butterfly reduction of v[16] across the warp: afterwards v[0] of lane l is
// the warp-wide sum of row l >> 1.
__device__ __forceinline__ float reduce16(float (&v)[kUnitRows]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool hi = lane & 16;
    const float send = hi ? v[i] : v[i + 8];
    const float keep = hi ? v[i + 8] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool hi = lane & 8;
    const float send = hi ? v[i] : v[i + 4];
    const float keep = hi ? v[i + 4] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool hi = lane & 4;
    const float send = hi ? v[i] : v[i + 2];
    const float keep = hi ? v[i + 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  {
    const bool hi = lane & 2;
    const float send = hi ? v[0] : v[1];
    const float keep = hi ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
  return v[0];
}

// Pre-scale of an activation feeding the next dequant-GEMV at input index k.
template <int QT>
__device__ __forceinline__ float pos_scale_inv(int k) {
  if (QT == COLI_Q_INT4_G128) {
    const int r = k & 7;
    const int p = r <= 4 ? r : r - 3;
    return __uint_as_float((uint32_t)(127 - 4 * p) << 23);
  }
  return (k & 1) ? (1.0f / 256.0f) : 1.0f;
}

// ------------------------------------------------------------------ one pass (nt tokens, all stages)

template <int QT, bool DOWN, int NT, int NTMAX>
__device__ __forceinline__ bool run_pass(const FwdArgs& a, int n_routed, int n_units, int stride, const Cursor& cons,
                                         Cursor& prod, uint8_t* wbuf, uint64_t* bars, int& stage, uint32_t& phase,
                                         uint64_t policy) {
  constexpr bool I4 = QT == COLI_Q_INT4_G128;
  constexpr int CODES = I4 ? 32 : 16;   // codes per lane per row per stage
  const int lane = threadIdx.x & 31;
  const int rows = rows_per_unit<DOWN>();
  const Unit u = cons.u;
  const DevExpert& ex = a.experts[u.slot];
  const int rbytes = row_bytes_of<QT>(u.K);
  const int G = u.K / 128, ZB = (G + 1) / 2;

  // this pass's tokens (input rows)
  const int p0 = u.pbeg + cons.pass * NTMAX;
  const int ntok = min(NT, u.cnt - cons.pass * NTMAX);
  const float* xrow[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int tt = t < ntok ? t : 0;
    xrow[t] = DOWN ? a.h + (size_t)(p0 + tt) * a.Fmax : a.xs + (size_t)a.pair_token[p0 + tt] * a.d;
  }
  // row r of the unit: gate/up rows rb*8 + (r & 7) of matrix r >> 3, or down row rb*16 + r
  float acc[NT][kUnitRows];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int r = 0; r < kUnitRows; ++r) acc[t][r] = 0.f;
  // int8: per-row zero-points (applied per stage) and scales (applied at the end)
  float z8[kUnitRows];
  if (!I4) {
#pragma unroll
    for (int r = 0; r < kUnitRows; ++r) {
      const int mat = DOWN ? 2 : (r >> 3);
      const int row = DOWN ? u.rb * kUnitRows + r : u.rb * 8 + (r & 7);
      z8[r] = (float)__ldg(ex.m[mat].z + row);
    }
  }

  bool ok = true;
  for (int kb = 0; kb < cons.n_kb; ++kb) {
    uint64_t* bar = bars + stage;
    const int kbyte = kb * kRowBytesPerStage + lane * 16;   // this lane's 16 bytes of each row
    const bool valid = kbyte < rbytes;
    const int code0 = I4 ? kbyte * 2 : kbyte;
    // scales / zero-points of the lane's group for the unit's rows (int4)
    float sc[kUnitRows], zc[kUnitRows];
    if constexpr (I4) {
      const int g = valid ? code0 / 128 : 0;
#pragma unroll
      for (int r = 0; r < kUnitRows; ++r) {
        const int mat = DOWN ? 2 : (r >> 3);
        const int row = DOWN ? u.rb * kUnitRows + r : u.rb * 8 + (r & 7);
        sc[r] = f16_bits_to_float(__ldg(static_cast<const uint16_t*>(ex.m[mat].s) + (size_t)row * G + g));
        const uint32_t zb = __ldg(ex.m[mat].z + (size_t)row * ZB + (g >> 1));
        zc[r] = (float)((g & 1) ? (zb >> 4) : (zb & 15u));
      }
    }
    if (!mbar_wait(bar, phase)) { ok = false; break; }
    if (valid) {
      const uint8_t* sbase = wbuf + stage * kStageBytes;
      const int half = lane >> 4, off = (lane & 15) * 16;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float xp[CODES];
#pragma unroll
        for (int i = 0; i < CODES; i += 4) {
          const float4 v = ldg_nc_f4(xrow[t] + code0 + i);
          xp[i] = v.x; xp[i + 1] = v.y; xp[i + 2] = v.z; xp[i + 3] = v.w;
        }
        float xsum = 0.f;   // sum of the unscaled activations of the lane's codes
#pragma unroll
        for (int i = 0; i < CODES; ++i)
          xsum = fmaf(xp[i], I4 ? int4_pos_scale(i) : ((i & 1) ? 256.f : 1.f), xsum);
#pragma unroll
        for (int r = 0; r < kUnitRows; ++r) {
          const int mat_slot = DOWN ? 0 : (r >> 3);
          const int rr = DOWN ? r : (r & 7);
          const uint4 w = lds128(smem_u32(sbase + (mat_slot * 2 + half) * rows * kBoxBytes + rr * kBoxBytes + off));
          float2 d2 = make_float2(0.f, 0.f);
          if constexpr (I4) {
            d2 = dot_word_int4(w.x, xp + 0, d2);
            d2 = dot_word_int4(w.y, xp + 8, d2);
            d2 = dot_word_int4(w.z, xp + 16, d2);
            d2 = dot_word_int4(w.w, xp + 24, d2);
            acc[t][r] = fmaf(sc[r], fmaf(-zc[r], xsum, d2.x + d2.y), acc[t][r]);
          } else {
            d2 = dot_word_int8(w.x, xp + 0, d2);
            d2 = dot_word_int8(w.y, xp + 4, d2);
            d2 = dot_word_int8(w.z, xp + 8, d2);
            d2 = dot_word_int8(w.w, xp + 12, d2);
            acc[t][r] += fmaf(-z8[r], xsum, d2.x + d2.y);
          }
        }
      }
    }
    __syncwarp();
    if (prod.valid) {
      if (lane == 0) {
        fence_proxy_async_smem();
        issue_stage<QT, DOWN>(a, prod, wbuf + stage * kStageBytes, bar, policy);
      }
      cursor_next<QT, DOWN, NTMAX>(a, n_routed, n_units, stride, prod);
    }
    if (++stage == kDecodeStages) { stage = 0; phase ^= 1u; }
  }
  if (!ok) return false;

#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const float v = reduce16(acc[t]);            // lane l: row l >> 1 of the unit
    const int r = lane >> 1;
    if (DOWN) {
      const int row = u.rb * kUnitRows + r;
      float val = v;
      if (!I4) val *= __ldg(static_cast<const float*>(ex.m[2].s) + row);
      if ((lane & 1) == 0 && t < ntok) a.y[(size_t)(p0 + t) * a.d + row] = val;
    } else {
      // lanes 0..15 hold gate rows 0..7, lanes 16..31 the same up rows
      const int row = u.rb * 8 + (r & 7);
      float val = v;
      if (!I4) val *= __ldg(static_cast<const float*>(ex.m[r >> 3].s) + row);
      const float upv = __shfl_down_sync(0xffffffffu, val, 16);
      if (lane < 16 && (lane & 1) == 0 && t < ntok) {
        const float hv = val / (1.0f + expf(-val)) * upv;
        a.h[(size_t)(p0 + t) * a.Fmax + row] = hv * pos_scale_inv<QT>(row);
      }
    }
  }
  return true;
}

template <int QT, bool DOWN, int NTMAX>
__global__ void __launch_bounds__(kDecodeWarps * 32, 1) decode_ffn_kernel(FwdArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t bars_all[kDecodeWarps][kDecodeStages];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wbuf = smem + (size_t)warp * kDecodeStages * kStageBytes;
  uint64_t* bars = bars_all[warp];

  const int n_routed = a.n_unique[0];
  const int n_units = n_units_of<DOWN>(a, n_routed);
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
  cursor_load<QT, DOWN, NTMAX>(a, n_routed, n_units, first, prod);
  cons = prod;
  for (int s = 0; s < kDecodeStages && prod.valid; ++s) {
    if (lane == 0) issue_stage<QT, DOWN>(a, prod, wbuf + s * kStageBytes, bars + s, policy);
    cursor_next<QT, DOWN, NTMAX>(a, n_routed, n_units, stride, prod);
  }
  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  while (cons.valid && ok) {
    const int ntok = min(NTMAX, cons.u.cnt - cons.pass * NTMAX);
    if (NTMAX == 1 || ntok <= 1)
      ok = run_pass<QT, DOWN, 1, NTMAX>(a, n_routed, n_units, stride, cons, prod, wbuf, bars, stage, phase, policy);
    else if (NTMAX == 2 || ntok <= 2)
      ok = run_pass<QT, DOWN, (NTMAX >= 2 ? 2 : 1), NTMAX>(a, n_routed, n_units, stride, cons, prod, wbuf, bars,
                                                          stage, phase, policy);
    else
      ok = run_pass<QT, DOWN, NTMAX, NTMAX>(a, n_routed, n_units, stride, cons, prod, wbuf, bars, stage, phase,
                                            policy);
    cons.kb = cons.n_kb - 1;
    cursor_next<QT, DOWN, NTMAX>(a, n_routed, n_units, stride, cons);
  }
  if (!ok) {
    if (lane == 0) set_status(a.status, COLI_DEV_WAIT_TIMEOUT);
    // drain: wait (bounded) for the stages still in flight before the CTA's
    // shared memory can be released
    for (int s = 0; s < kDecodeStages; ++s) {
      const int st = (stage + s) % kDecodeStages;
      const uint32_t ph = phase ^ ((stage + s) >= kDecodeStages ? 1u : 0u);
      mbar_wait(bars + st, ph);
    }
  }
}

template <int QT, bool DOWN, int NTMAX>
static cudaError_t launch_decode_t(const FwdArgs& a, cudaStream_t st, int num_sms) {
  const size_t smem = (size_t)kDecodeWarps * kDecodeStages * kStageBytes + 1024;
  auto kern = decode_ffn_kernel<QT, DOWN, NTMAX>;
  static bool attr_set = false;   // per template instance
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<num_sms, kDecodeWarps * 32, smem, st>>>(a);
  return cudaGetLastError();
}

template <bool DOWN>
static cudaError_t launch_decode(const FwdArgs& a, int max_tok, cudaStream_t st, int num_sms) {
  const bool i4 = a.qtype == COLI_Q_INT4_G128;
  if (max_tok <= 1)
    return i4 ? launch_decode_t<COLI_Q_INT4_G128, DOWN, 1>(a, st, num_sms)
              : launch_decode_t<COLI_Q_INT8_PC, DOWN, 1>(a, st, num_sms);
  if (max_tok <= 2)
    return i4 ? launch_decode_t<COLI_Q_INT4_G128, DOWN, 2>(a, st, num_sms)
              : launch_decode_t<COLI_Q_INT8_PC, DOWN, 2>(a, st, num_sms);
  return i4 ? launch_decode_t<COLI_Q_INT4_G128, DOWN, 4>(a, st, num_sms)
            : launch_decode_t<COLI_Q_INT8_PC, DOWN, 4>(a, st, num_sms);
}

cudaError_t launch_decode_gateup(const FwdArgs& a, int max_tok, cudaStream_t st, int num_sms) {
  return launch_decode<false>(a, max_tok, st, num_sms);
}

cudaError_t launch_decode_down(const FwdArgs& a, int max_tok, cudaStream_t st, int num_sms) {
  return launch_decode<true>(a, max_tok, st, num_sms);
}

}  // namespace coli
