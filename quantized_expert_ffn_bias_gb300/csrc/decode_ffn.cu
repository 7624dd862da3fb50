// Expert FFN for small token counts (decode, MTP verify): HBM-bound dequant-GEMV.
//
// Each chosen expert's packed weights are streamed once per call for all the
// tokens routed to it (batch-union grouping, "25GB RAM runs 744B GLM-5.2" page
// (pwwt.cn), section 3.4) and dequantised as (code - zero_point) * scale
// ("Colibri walkthrough" page (discosf.com), section 3.4).
//
// Work unit = one warp and 16 matrix rows: 8 rows of gate with the same 8 rows
// of up (SwiGLU needs both), or 16 rows of down.  A pipeline stage holds 512
// bytes of each of the 16 rows (TMA boxes of 256 bytes); lane l owns bytes
// [16l, 16l+16) of every row, i.e. 32 int4 or 16 int8 codes.  The lane's
// activations are loaded once per stage (prefetched one stage ahead) and
// reused for all 16 rows, which also give 16 independent accumulation chains.
// A butterfly reduction across the warp ends the unit.  Each warp runs its own
// kDecodeStages-deep mbarrier pipeline; every wait is bounded and a timeout
// sets the workspace status word.
//
// Per (row, group) the scale s and the zero point z enter once:
// s*sum((c - z) x) = s*(sum(c x) - z*sum(x)).  The (s, z) pairs of the stage's
// groups are built cooperatively in a 1 KB table per warp.
//
// int4 (integer dot products): the activations enter in 16-bit fixed point per
// block of 32 inputs, x = sx*(256*hi + lo) with hi a signed and lo an unsigned
// byte, prepared once per token (gate/up: by the routing kernel) or per pair row
// (down: by quantize_h after the gate/up kernel).  Masking a word
// of codes and its 4-bit shift with 0x0F0F0F0F gives the even and odd codes as
// bytes, so one 8-code word costs three logic ops and four dp4a; sum(c*q) and
// z*sum(q) are exact integers and one conversion per 32 codes brings them to
// fp32.  The fixed point keeps every input to within 2^-16 of its block's
// largest magnitude.
//
// Integer-dot inputs (IDOT, both weight types): the activations enter as int8
// codes q per block of 32 with the block scale 2^(e-6) (warp_quantize_block32_i8);
// int4 weights take four dp4a per 8-code word pair as above but on one byte
// plane, int8 weights four dp4a per 16 codes (u8 codes times s8 activations);
// sum((c - z) q) stays an exact integer and one conversion per block half
// brings it to fp32.
//
// int8 (exact fp32): a code c placed at mantissa bit 4p (int4)
// or 8p (int8) of the float 2^23 gives 2^23 + c*16^p; subtracting 2^23 leaves
// c*16^p exactly, and the activation was pre-multiplied by 16^-p (an exact
// power of two), so the product is c*x; sum(x) is precomputed per block.
#include "moe_internal.cuh"

namespace coli {

constexpr int kRows = 16;                                     // rows per warp unit
constexpr int kRowBytesPerStage = 512;
constexpr int kBoxBytes = kTmaBoxBytes;
constexpr int kStageBytes = kRows * kRowBytesPerStage;        // 8 KB
constexpr int kGroupsPerStage = 8;                            // int4: 1024 codes per row per stage
constexpr int kMaxNT = 2;                                     // tokens per pass (more: further passes)

static_assert(kGateUpBoxRows == kRows / 2 && kDownBoxRows == kRows, "TMA boxes must match the unit rows");

struct Unit {
  int slot;   // storage slot of the expert's weights (its id unless an expert cache maps it)
  int rb;     // row block: gate/up rows rb*8.., down rows rb*16..
  int pbeg;   // first grouped pair row of the expert
  int cnt;    // tokens routed to the expert
  int K;      // inputs of the streamed matrix
};

template <bool DOWN>
__device__ __forceinline__ int block_rows() { return DOWN ? kRows : kRows / 2; }

template <bool DOWN>
__device__ __forceinline__ bool get_unit(const FwdArgs& a, int u, int n_routed, Unit& out) {
  // the shared expert's units first (it carries every token), then the routed experts' in unit-table
  // order (most tokens first)
  const int rows = block_rows<DOWN>();
  const int per_routed = (DOWN ? a.d : a.F) / rows;
  const int per_shared = a.has_shared ? (DOWN ? a.d : a.Fs) / rows : 0;
  int i, rb;
  if (u < per_shared) {
    i = n_routed;
    rb = u;
  } else {
    u -= per_shared;
    if (u >= n_routed * per_routed) return false;
    i = u / per_routed;
    rb = u % per_routed;
  }
  const int4 e = __ldcg(a.utab + i);      // (expert, first pair row, pairs), written by the routing kernel
  out.slot = a.slot_of ? __ldg(a.slot_of + e.x) : e.x;   // where the expert's weights are stored
  out.rb = rb;
  out.pbeg = e.y;
  out.cnt = e.z;
  out.K = DOWN ? (e.x == a.E ? a.Fs : a.F) : a.d;
  return true;
}

template <bool DOWN>
__device__ __forceinline__ int n_units_of(const FwdArgs& a, int n_routed) {
  const int rows = block_rows<DOWN>();
  const int per_routed = (DOWN ? a.d : a.F) / rows;
  const int per_shared = a.has_shared ? (DOWN ? a.d : a.Fs) / rows : 0;
  return n_routed * per_routed + per_shared;
}

template <int QT>
__device__ __forceinline__ int row_bytes_of(int K) { return QT == COLI_Q_INT4_G128 ? K / 2 : K; }

// Cursor over a warp's (unit, pass, stage) sequence.
struct Cursor {
  int unit, pass, kb, n_kb, n_pass;
  bool valid;
  Unit u;
};

template <int QT, bool DOWN>
__device__ __forceinline__ void cursor_load(const FwdArgs& a, int n_routed, int n_units, int unit, Cursor& c) {
  c.unit = unit;
  c.pass = 0;
  c.kb = 0;
  c.valid = unit < n_units && get_unit<DOWN>(a, unit, n_routed, c.u);
  if (c.valid) {
    c.n_kb = (row_bytes_of<QT>(c.u.K) + kRowBytesPerStage - 1) / kRowBytesPerStage;
    c.n_pass = (c.u.cnt + kMaxNT - 1) / kMaxNT;
    c.valid = c.n_pass > 0;
  }
}

template <int QT, bool DOWN>
__device__ __forceinline__ void cursor_next(const FwdArgs& a, int n_routed, int n_units, int stride, Cursor& c) {
  if (++c.kb < c.n_kb) return;
  c.kb = 0;
  if (++c.pass < c.n_pass) return;
  cursor_load<QT, DOWN>(a, n_routed, n_units, c.unit + stride, c);
}

// Shared layout of a stage.  gate/up: [matrix][box][8 rows][boxw]; down: [box][16 rows][boxw]
// (boxw = 256, or the row length for 128-byte rows).
template <bool DOWN>
__device__ __forceinline__ int stage_off(int r, int box, int boxw) {
  return DOWN ? box * 4096 + r * boxw : (r >> 3) * 4096 + box * 2048 + (r & 7) * boxw;
}

template <int QT, bool DOWN>
__device__ __forceinline__ void issue_stage(const FwdArgs& a, const Cursor& c, uint8_t* stage, uint64_t* bar,
                                            uint64_t policy) {
  const int rb_bytes = row_bytes_of<QT>(c.u.K);
  const int boxw = rb_bytes < kBoxBytes ? rb_bytes : kBoxBytes;
  const int x0 = c.kb * kRowBytesPerStage;
  const int nbox = x0 + kBoxBytes < rb_bytes ? 2 : 1;
  mbar_arrive_expect_tx(bar, (uint32_t)(kRows * nbox * boxw));
  if (DOWN) {
    const CUtensorMap* map = a.maps + (size_t)c.u.slot * 3 + 2;
    for (int b = 0; b < nbox; ++b)
      tma_load_2d(stage + stage_off<true>(0, b, boxw), map, x0 + b * kBoxBytes, c.u.rb * kRows, bar, policy);
  } else {
    for (int m = 0; m < 2; ++m) {
      const CUtensorMap* map = a.maps + (size_t)c.u.slot * 3 + m;
      for (int b = 0; b < nbox; ++b)
        tma_load_2d(stage + stage_off<false>(m * 8, b, boxw), map, x0 + b * kBoxBytes, c.u.rb * 8, bar, policy);
    }
  }
}

__device__ __forceinline__ float f16_bits_to_float(uint32_t b) {
  return __half2float(__ushort_as_half((unsigned short)b));
}

// The packed dequant-dot of one 32-bit word of int8 codes (PTX text): codes at
// mantissa positions, minus the magic pair %M, times two activation pairs.
#define COLI_WORD8(Q, X01, X23, M, FIRST)                                 \
  "shr.b32 v, " Q ", 16;\n\t"                                             \
  "lop3.b32 a0, " Q ", 0x000000FF, 0x4B000000, 0xEA;\n\t"                 \
  "lop3.b32 a1, " Q ", 0x0000FF00, 0x4B000000, 0xEA;\n\t"                 \
  "lop3.b32 a2, v, 0x000000FF, 0x4B000000, 0xEA;\n\t"                     \
  "lop3.b32 a3, v, 0x0000FF00, 0x4B000000, 0xEA;\n\t"                     \
  "mov.b64 p0, {a0, a1};\n\tmov.b64 p1, {a2, a3};\n\t"                    \
  "sub.rn.f32x2 p0, p0, " M ";\n\tsub.rn.f32x2 p1, p1, " M ";\n\t"        \
  FIRST                                                                   \
  "fma.rn.f32x2 %0, p1, " X23 ", %0;\n\t"

// One row slice of 16 int8 codes against 16 pre-scaled activations (8 pairs).
__device__ __forceinline__ uint64_t dot_row_int8(uint4 w, const ulonglong2 (&x)[8], uint64_t m2) {
  uint64_t acc;
  asm("{\n\t"
      ".reg .b32 v, a0, a1, a2, a3;\n\t"
      ".reg .b64 p0, p1;\n\t"
      COLI_WORD8("%1", "%5", "%6", "%13", "mul.rn.f32x2 %0, p0, %5;\n\t")
      COLI_WORD8("%2", "%7", "%8", "%13", "fma.rn.f32x2 %0, p0, %7, %0;\n\t")
      COLI_WORD8("%3", "%9", "%10", "%13", "fma.rn.f32x2 %0, p0, %9, %0;\n\t")
      COLI_WORD8("%4", "%11", "%12", "%13", "fma.rn.f32x2 %0, p0, %11, %0;\n\t")
      "}"
      : "=l"(acc)
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "l"(x[0].x), "l"(x[0].y), "l"(x[1].x), "l"(x[1].y), "l"(x[2].x),
        "l"(x[2].y), "l"(x[3].x), "l"(x[3].y), "l"(m2));
  return acc;
}
#undef COLI_WORD8

// One row slice of 32 int4 codes against the lane's fixed-point activations:
// xh[8] / xl[8] = hi / lo bytes in unpack order.  Returns sum(c * q) exactly.
__device__ __forceinline__ int dot_row_int4_dp4a(uint4 w, const uint32_t (&xh)[8], const uint32_t (&xl)[8]) {
  int hi = 0;
  uint32_t lo = 0;
  const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t ev = q[j] & 0x0F0F0F0Fu, od = (q[j] >> 4) & 0x0F0F0F0Fu;
    asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(hi) : "r"(ev), "r"(xh[2 * j]));
    asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(hi) : "r"(od), "r"(xh[2 * j + 1]));
    asm("dp4a.u32.u32 %0, %1, %2, %0;" : "+r"(lo) : "r"(ev), "r"(xl[2 * j]));
    asm("dp4a.u32.u32 %0, %1, %2, %0;" : "+r"(lo) : "r"(od), "r"(xl[2 * j + 1]));
  }
  return hi * 256 + (int)lo;
}

// The same with int8 activation codes (one byte plane): returns sum(c * q) exactly.
__device__ __forceinline__ int dot_row_int4_i8(uint4 w, const uint32_t (&xq)[8]) {
  int acc = 0;
  const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t ev = q[j] & 0x0F0F0F0Fu, od = (q[j] >> 4) & 0x0F0F0F0Fu;
    asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(ev), "r"(xq[2 * j]));
    asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(od), "r"(xq[2 * j + 1]));
  }
  return acc;
}

// 16 int8 weight codes (u8, natural order) against 16 int8 activation codes: sum(c * q) exactly.
__device__ __forceinline__ int dot_row_int8_i8(uint4 w, const uint32_t (&xq)[4]) {
  int acc = 0;
  asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(w.x), "r"(xq[0]));
  asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(w.y), "r"(xq[1]));
  asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(w.z), "r"(xq[2]));
  asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(w.w), "r"(xq[3]));
  return acc;
}

__device__ __forceinline__ float pair_sum(uint64_t p) {
  return __uint_as_float((uint32_t)p) + __uint_as_float((uint32_t)(p >> 32));
}

__device__ __forceinline__ ulonglong2 ldg_nc_u64x2(const float* p) {
  ulonglong2 v;
  asm volatile("ld.global.nc.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p));
  return v;
}

// Butterfly reduction of v[16] across the warp: afterwards v[0] of lane l is
// the warp-wide sum of row l >> 1.
__device__ __forceinline__ float reduce16(float (&v)[kRows]) {
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

// row r of the unit -> (matrix, matrix row)
template <bool DOWN>
__device__ __forceinline__ void unit_row(const Unit& u, int r, int& mat, int& row) {
  if (DOWN) { mat = 2; row = u.rb * kRows + r; }
  else { mat = r >> 3; row = u.rb * 8 + (r & 7); }
}

// Raw (scale, zero-point) data of one stage for the (row, 4 groups) a lane fills
// in the stage table: lane l covers row l >> 1 and groups 4*(l & 1) .. +3.
struct ScaleRaw {
  uint32_t s01, s23;   // four fp16 scales
  uint32_t z4;         // four zero nibbles in the low 16 bits
};

template <bool DOWN>
__device__ __forceinline__ ScaleRaw load_scales_int4(const DevExpert& ex, const Unit& u, int kb, int G) {
  const int lane = threadIdx.x & 31;
  const int r = lane >> 1;
  const int g0 = kb * kGroupsPerStage + 4 * (lane & 1);
  int mat, row;
  unit_row<DOWN>(u, r, mat, row);
  const DevMat& M = ex.m[mat];
  const uint16_t* s = static_cast<const uint16_t*>(M.s) + (size_t)row * G + g0;
  const uint8_t* z = M.z + (size_t)row * ((G + 1) / 2) + g0 / 2;
  ScaleRaw o;
  if ((G & 3) == 0 && (reinterpret_cast<uintptr_t>(M.s) & 7) == 0 && (reinterpret_cast<uintptr_t>(M.z) & 1) == 0 &&
      g0 < G) {
    // the lane's four scales are 8 aligned bytes and its four zero-point nibbles 2 aligned bytes:
    // two loads instead of six (these loads sit on every stage of every warp)
    const uint2 s4 = __ldg(reinterpret_cast<const uint2*>(s));
    o.s01 = s4.x;
    o.s23 = s4.y;
    o.z4 = __ldg(reinterpret_cast<const uint16_t*>(z));
    return o;
  }
  uint32_t sv[4], zv[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) sv[i] = g0 + i < G ? __ldg(s + i) : 0u;
#pragma unroll
  for (int i = 0; i < 2; ++i) zv[i] = g0 + 2 * i < G ? __ldg(z + i) : 0u;
  o.s01 = sv[0] | (sv[1] << 16);
  o.s23 = sv[2] | (sv[3] << 16);
  o.z4 = zv[0] | (zv[1] << 8);
  return o;
}

// Write the lane's four entries of the stage table [16 rows][8 groups]:
// (s, s*z) for the fp32 path, (s, z as int bits) for the integer path.
template <bool DP>
__device__ __forceinline__ void store_scales_int4(float2* tab, const ScaleRaw& o) {
  const int lane = threadIdx.x & 31;
  float2* dst = tab + (lane >> 1) * kGroupsPerStage + 4 * (lane & 1);
  const uint32_t sv[4] = {o.s01 & 0xFFFFu, o.s01 >> 16, o.s23 & 0xFFFFu, o.s23 >> 16};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float s = f16_bits_to_float(sv[i]);
    const int zi = (int)((o.z4 >> (4 * i)) & 15u);
    dst[i] = DP ? make_float2(s, __int_as_float(zi)) : make_float2(s, s * (float)zi);
  }
}

// ------------------------------------------------------------------ one pass (NT tokens, all stages)

template <int QT, bool DOWN, int NT, bool ID>
__device__ __forceinline__ bool run_pass(const FwdArgs& a, int n_routed, int n_units, int stride, const Cursor& cons,
                                         Cursor& prod, uint8_t* wbuf, uint64_t* bars, float2* tab, int& stage,
                                         uint32_t& phase, uint64_t policy) {
  constexpr bool I4 = QT == COLI_Q_INT4_G128;
  constexpr bool DP = I4 || ID;         // integer dot products (fixed-point or int8 activations)
  constexpr int CODES = I4 ? 32 : 16;   // codes per lane per row per stage
  constexpr int XQ = CODES / 4;         // 16-byte activation loads per token
  const int lane = threadIdx.x & 31;
  const Unit u = cons.u;
  const DevExpert& ex = a.experts[u.slot];
  const int rbytes = row_bytes_of<QT>(u.K);
  const int boxw = rbytes < kBoxBytes ? rbytes : kBoxBytes;
  const int G = u.K / 128;

  // this pass's input rows and their block sums
  const int p0 = u.pbeg + cons.pass * kMaxNT;
  const int ntok = min(NT, u.cnt - cons.pass * kMaxNT);
  const float* xrow[NT];
  const float* srow[NT];
  const uint32_t* qrow[NT];
  const int2* qsrow[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int tt = t < ntok ? t : 0;
    if (DOWN) {
      xrow[t] = a.h + (size_t)(p0 + tt) * a.Fmax;
      srow[t] = a.hsum + (size_t)(p0 + tt) * (a.Fmax / 8);
      qrow[t] = a.hq + (size_t)(p0 + tt) * (a.Fmax / 2);
      qsrow[t] = a.hqs + (size_t)(p0 + tt) * (a.Fmax / kXqBlock);
    } else {
      const int tok = a.pair_token[p0 + tt];
      xrow[t] = a.xs + (size_t)tok * a.d;
      srow[t] = a.xsum + (size_t)tok * (a.d / kXsumBlock);
      qrow[t] = a.xq + (size_t)tok * (a.d / 2);
      qsrow[t] = a.xqs + (size_t)tok * (a.d / kXqBlock);
    }
  }
  auto code0_of = [&](int kb) {
    const int kbyte = kb * kRowBytesPerStage + lane * 16;
    return kbyte < rbytes ? (I4 ? kbyte * 2 : kbyte) : -1;
  };
  auto load_x = [&](int t, int code0, ulonglong2 (&xq)[8], float& xsum) {
    const int c = code0 < 0 ? 0 : code0;
    if constexpr (DP) {   // 64 bytes of hi/lo words (as 4 x 16 bytes) and the block's (sx, sum q);
                          // int8 codes: the 32 bytes of the block (int4) or the lane's 16 (int8)
      const int b = c / kXqBlock;
      const ulonglong2* src = reinterpret_cast<const ulonglong2*>(qrow[t] + (size_t)b * 16);
      if constexpr (ID && !I4) {
        xq[0] = __ldg(src + (c % kXqBlock) / 16);
      } else {
#pragma unroll
        for (int i = 0; i < (ID ? 2 : 4); ++i) xq[i] = __ldg(src + i);
      }
      const int2 qs = __ldg(qsrow[t] + b);
      xq[4].x = (unsigned long long)(uint32_t)qs.x | ((unsigned long long)(uint32_t)qs.y << 32);
      return;
    } else {
#pragma unroll
      for (int i = 0; i < XQ; ++i) xq[i] = ldg_nc_u64x2(xrow[t] + c + 4 * i);
    if (DOWN) {          // sums of h over 8 consecutive inputs
      if (I4) {
        const float4 h4 = __ldg(reinterpret_cast<const float4*>(srow[t] + c / 8));
        xsum = (h4.x + h4.y) + (h4.z + h4.w);
      } else {
        const float2 h2 = __ldg(reinterpret_cast<const float2*>(srow[t] + c / 8));
        xsum = h2.x + h2.y;
      }
    } else {             // sums of x over blocks of 16 inputs
      if (I4) {
        const float2 s2 = __ldg(reinterpret_cast<const float2*>(srow[t] + c / kXsumBlock));
        xsum = s2.x + s2.y;
      } else {
        xsum = __ldg(srow[t] + c / kXsumBlock);
      }
    }
    }
  };

  // int8: the (s, s*z) of the unit's 16 rows, once per pass
  if (!I4) {
    __syncwarp();
    if (lane < kRows) {
      int mat, row;
      unit_row<DOWN>(u, lane, mat, row);
      const float s = __ldg(static_cast<const float*>(ex.m[mat].s) + row);
      const int z = __ldg(ex.m[mat].z + row);
      tab[lane] = make_float2(s, ID ? __int_as_float(z) : s * (float)z);
    }
    __syncwarp();
  }

  float acc[NT][kRows];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int r = 0; r < kRows; ++r) acc[t][r] = 0.f;

  const uint64_t m2 = 0x4B0000004B000000ull;   // (2^23, 2^23)
  // activations of the first token and scales, loaded two stages ahead
  ulonglong2 xq0[8], xq1[8];
  float xs0 = 0.f, xs1 = 0.f;
  ScaleRaw sr = {0u, 0u, 0u}, sr1 = {0u, 0u, 0u};
  load_x(0, code0_of(0), xq0, xs0);
  if (I4) sr = load_scales_int4<DOWN>(ex, u, 0, G);
  if (cons.n_kb > 1) {
    load_x(0, code0_of(1), xq1, xs1);
    if (I4) sr1 = load_scales_int4<DOWN>(ex, u, 1, G);
  }

  bool ok = true;
  for (int kb = 0; kb < cons.n_kb; ++kb) {
    const int code0 = code0_of(kb);
    if (I4) {                       // stage table of (s, s*z) or (s, z)
      __syncwarp();
      store_scales_int4<DP>(tab, sr);
      __syncwarp();
    }
    // current-stage activations (token 0 prefetched); rotate and prefetch stage kb + 2
    ulonglong2 xq[8];
    float xsum = xs0;
#pragma unroll
    for (int i = 0; i < 8; ++i) { xq[i] = xq0[i]; xq0[i] = xq1[i]; }
    xs0 = xs1;
    sr = sr1;
    if (kb + 2 < cons.n_kb) {
      load_x(0, code0_of(kb + 2), xq1, xs1);
      if (I4) sr1 = load_scales_int4<DOWN>(ex, u, kb + 2, G);
    }
    const int g = I4 ? (code0 < 0 ? 0 : (code0 >> 7) - kb * kGroupsPerStage) : 0;
    if (!mbar_wait(bars + stage, phase, a.wait_ns)) { ok = false; break; }
    if (code0 >= 0) {
      const uint8_t* sbase = wbuf + stage * kStageBytes + (lane & 15) * 16;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t > 0) load_x(t, code0, xq, xsum);
        if constexpr (ID && !I4) {
          const uint32_t xw[4] = {(uint32_t)xq[0].x, (uint32_t)(xq[0].x >> 32), (uint32_t)xq[0].y,
                                  (uint32_t)(xq[0].y >> 32)};
          const float sx = __uint_as_float((uint32_t)xq[4].x);
          int qs16 = 0;                              // sum of the lane's 16 codes
#pragma unroll
          for (int j = 0; j < 4; ++j) asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(qs16) : "r"(0x01010101u), "r"(xw[j]));
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            const uint4 w = lds128(smem_u32(sbase + stage_off<DOWN>(r, lane >> 4, boxw)));
            const float2 sz = tab[r];
            const int comb = dot_row_int8_i8(w, xw) - __float_as_int(sz.y) * qs16;
            acc[t][r] = fmaf(sz.x * sx, (float)comb, acc[t][r]);
          }
        } else if (DP) {
          uint32_t xh[8], xl[8];
          float sx;
          int qsum;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            xh[4 * i] = (uint32_t)xq[i].x; xh[4 * i + 1] = (uint32_t)(xq[i].x >> 32);
            xh[4 * i + 2] = (uint32_t)xq[i].y; xh[4 * i + 3] = (uint32_t)(xq[i].y >> 32);
            xl[4 * i] = (uint32_t)xq[2 + i].x; xl[4 * i + 1] = (uint32_t)(xq[2 + i].x >> 32);
            xl[4 * i + 2] = (uint32_t)xq[2 + i].y; xl[4 * i + 3] = (uint32_t)(xq[2 + i].y >> 32);
          }
          sx = __uint_as_float((uint32_t)xq[4].x);
          qsum = (int)(uint32_t)(xq[4].x >> 32);
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            const uint4 w = lds128(smem_u32(sbase + stage_off<DOWN>(r, lane >> 4, boxw)));
            const float2 sz = tab[r * kGroupsPerStage + g];
            const int comb = (ID ? dot_row_int4_i8(w, xh) : dot_row_int4_dp4a(w, xh, xl)) -
                             __float_as_int(sz.y) * qsum;
            acc[t][r] = fmaf(sz.x * sx, (float)comb, acc[t][r]);
          }
        } else {
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            const uint4 w = lds128(smem_u32(sbase + stage_off<DOWN>(r, lane >> 4, boxw)));
            const float2 sz = I4 ? tab[r * kGroupsPerStage + g] : tab[r];
            const uint64_t d2 = dot_row_int8(w, xq, m2);
            acc[t][r] = fmaf(sz.x, pair_sum(d2), fmaf(-sz.y, xsum, acc[t][r]));
          }
        }
      }
    }
    __syncwarp();
    if (prod.valid) {
      if (lane == 0) {
        fence_proxy_async_smem();
        issue_stage<QT, DOWN>(a, prod, wbuf + stage * kStageBytes, bars + stage, policy);
      }
      cursor_next<QT, DOWN>(a, n_routed, n_units, stride, prod);
    }
    if (++stage == kDecodeStages) { stage = 0; phase ^= 1u; }
  }
  if (!ok) return false;

#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const float v = reduce16(acc[t]);           // lane l: row l >> 1 of the unit
    if (DOWN) {
      const int row = u.rb * kRows + (lane >> 1);
      if ((lane & 1) == 0 && t < ntok) a.y[(size_t)(p0 + t) * a.d + row] = v;
    } else {
      // lanes 0..15: gate rows 0..7, lanes 16..31: the same up rows
      const float up = __shfl_down_sync(0xffffffffu, v, 16);
      const float hv = v / (1.0f + expf(-v)) * up;          // silu(gate) * up
      float hs = hv;                                           // sum of the 8 rows (lanes 0, 2, .., 14)
      if constexpr (!I4 && !ID) {
        hs += __shfl_xor_sync(0xffffffffu, hs, 2);
        hs += __shfl_xor_sync(0xffffffffu, hs, 4);
        hs += __shfl_xor_sync(0xffffffffu, hs, 8);
      }
      const int row = u.rb * 8 + (lane >> 1);
      // int4 and integer-dot inputs: plain h (quantize_h converts it for the down kernel);
      // int8: pre-scaled h and its sums
      if (lane < 16 && (lane & 1) == 0 && t < ntok)
        a.h[(size_t)(p0 + t) * a.Fmax + row] = (I4 || ID) ? hv : hv * act_prescale(QT, row);
      if (!I4 && !ID && lane == 0 && t < ntok) a.hsum[(size_t)(p0 + t) * (a.Fmax / 8) + u.rb] = hs;
    }
  }
  return true;
}

template <int QT, bool DOWN, int NTMAX, bool ID>
__global__ void __launch_bounds__(kDecodeWarps * 32, 1) decode_ffn_kernel(FwdArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t bars_all[kDecodeWarps][kDecodeStages];
  __shared__ float2 tabs[kDecodeWarps][kRows * kGroupsPerStage];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wbuf = smem + (size_t)warp * kDecodeStages * kStageBytes;
  uint64_t* bars = bars_all[warp];
  float2* tab = tabs[warp];

  griddep_launch_dependents();
  griddep_wait();                  // routing (gate/up) or h (down) of the previous kernel
  const int n_routed = a.n_unique[0];
  const int n_units = n_units_of<DOWN>(a, n_routed);
  const int stride = gridDim.x * kDecodeWarps;
  // units are dealt warp-major over the CTAs, so that a last, partial round of units keeps
  // every SM streaming (5 or 6 warps each) instead of filling some SMs and idling others
  const int first = warp * gridDim.x + blockIdx.x;
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
    // failure-path test: warp 0 of CTA 0 withholds its first gate/up stage, so its wait reaches the
    // (shortened) wait limit and the warp stops with the status set
    const bool withhold = !DOWN && s == 0 && blockIdx.x == 0 && warp == 0 && (a.inject & COLI_INJECT_WITHHOLD_STAGE);
    if (lane == 0 && !withhold) issue_stage<QT, DOWN>(a, prod, wbuf + s * kStageBytes, bars + s, policy);
    cursor_next<QT, DOWN>(a, n_routed, n_units, stride, prod);
  }
  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  while (cons.valid && ok) {
    const int ntok = min(kMaxNT, cons.u.cnt - cons.pass * kMaxNT);
    if (NTMAX == 1 || ntok <= 1)
      ok = run_pass<QT, DOWN, 1, ID>(a, n_routed, n_units, stride, cons, prod, wbuf, bars, tab, stage, phase,
                                     policy);
    else
      ok = run_pass<QT, DOWN, (NTMAX >= 2 ? 2 : 1), ID>(a, n_routed, n_units, stride, cons, prod, wbuf, bars, tab,
                                                       stage, phase, policy);
    cons.kb = cons.n_kb - 1;
    cursor_next<QT, DOWN>(a, n_routed, n_units, stride, cons);
  }
  if (!ok) {
    if (lane == 0) {
      set_status(a.status, COLI_DEV_WAIT_TIMEOUT);
      // drain: wait (bounded) for the stages that may still have a copy in flight
      for (int s = 0; s < kDecodeStages; ++s) mbar_wait(bars + s, phase ^ (s < stage ? 1u : 0u), a.wait_ns);
    }
    __syncwarp();
  }
}

template <int QT, bool DOWN, int NTMAX, bool ID>
static cudaError_t launch_decode_t(const FwdArgs& a, cudaStream_t st, int num_sms) {
  const size_t smem = (size_t)kDecodeWarps * kDecodeStages * kStageBytes + 1024;
  auto kern = decode_ffn_kernel<QT, DOWN, NTMAX, ID>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(num_sms), dim3(kDecodeWarps * 32), smem, st, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <bool DOWN, bool ID>
static cudaError_t launch_decode_id(const FwdArgs& a, int max_tok, cudaStream_t st, int num_sms) {
  const bool i4 = a.qtype == COLI_Q_INT4_G128;
  if (max_tok <= 1)
    return i4 ? launch_decode_t<COLI_Q_INT4_G128, DOWN, 1, ID>(a, st, num_sms)
              : launch_decode_t<COLI_Q_INT8_PC, DOWN, 1, ID>(a, st, num_sms);
  return i4 ? launch_decode_t<COLI_Q_INT4_G128, DOWN, 2, ID>(a, st, num_sms)
            : launch_decode_t<COLI_Q_INT8_PC, DOWN, 2, ID>(a, st, num_sms);
}

template <bool DOWN>
static cudaError_t launch_decode(const FwdArgs& a, int max_tok, cudaStream_t st, int num_sms) {
  return a.idot ? launch_decode_id<DOWN, true>(a, max_tok, st, num_sms)
                : launch_decode_id<DOWN, false>(a, max_tok, st, num_sms);
}

cudaError_t launch_decode_gateup(const FwdArgs& a, int max_tok, cudaStream_t st, int num_sms) {
  return launch_decode<false>(a, max_tok, st, num_sms);
}

cudaError_t launch_decode_down(const FwdArgs& a, int max_tok, cudaStream_t st, int num_sms) {
  return launch_decode<true>(a, max_tok, st, num_sms);
}

}  // namespace coli
