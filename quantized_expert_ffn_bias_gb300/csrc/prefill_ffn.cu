// Expert FFN for large token counts (prefill, batched verification): grouped
// GEMMs on the 5th-generation tensor cores (tcgen05, accumulators in TMEM).
//
// Each chosen expert's weights are dequantised once per chunk of up to 128 of
// its tokens (batch-union grouping, "25GB RAM runs 744B GLM-5.2" page
// (pwwt.cn), section 3.4) and multiplied with those tokens' activations:
//   gate/up: D[n][t] = sum_k W[n][k] * X[t][k] for 128 weight rows n (MMA M =
//            128) and the chunk's tokens t (MMA N = tokens rounded up to 16),
//            gate and up into two TMEM accumulators; SwiGLU in the epilogue;
//   down:    D[m][t] = sum_n Wd[m][n] * H[t][n].
// Weights w = (code - zero_point) * scale ("Colibri walkthrough" page
// (discosf.com), section 3.4) are produced as fp16 by dequantising warps
// (int4: fp16((c - z) * s), one rounding; int8: exact c - z with the row scale
// applied in the epilogue).  Activations are fp16: bf16 values convert
// exactly in fp16's normal range, and fp16 keeps 11 significant bits of the
// dequantised weights where bf16 would keep 8.
//
// The dequantised weight tile is the MMA's A operand and lives in tensor
// memory (written with tcgen05.st), so shared memory only carries the raw
// codes and the activation tiles; with small N an A operand in shared memory
// would be re-read by every MMA and shared-memory bandwidth would set the pace.
//
// int4 unpacking: a 32-bit word holds 8 codes n0..n7 (code i in bits 4i..4i+3).
// Masking the word and its 8-bit shift with 0x000F000F (into fp16 1024 + c)
// and with 0x00F000F0 (into fp16 64 + c) gives the pairs (n0,n4), (n1,n5),
// (n2,n6), (n3,n7) with one shift and four logic ops, so within every group of
// 8 inputs the A operand holds the codes in the order 0,4,1,5,2,6,3,7.  The activation matrices (X for gate/up, H for down) are
// stored with the same permutation inside each group of 8 columns, which
// leaves every dot product unchanged.  int8 keeps the natural order.
//
// CTA (persistent, one per SM): warp 0 issues TMA loads (raw codes and
// activation rows) into a ring of stages, with L2 prefetch of the codes further
// ahead; warp 1 owns TMEM and issues the MMAs (one thread; for gate/up it
// issues the gate matrix and warp 22 the up matrix: the issuing thread sets the
// pace, and two of them on different sub-partitions issue more MMAs); warps
// 2..5 run the epilogue; warps 6..21 dequantise into a ring of TMEM A stages.
// Every CTA loads its own activation tiles with plain TMA loads.
// All waits are bounded; a timeout sets the status word and every role stops.
#include <algorithm>

#include "moe_internal.cuh"

namespace coli {

constexpr int kPfM = 128;           // weight rows per tile (MMA M, TMEM lanes)
constexpr int kPfN = kPrefillChunk;  // tokens per chunk (largest MMA N)
constexpr int kPfBBox = kPrefillBBox;   // activation rows per TMA box
constexpr int kPfEpWarps = 4;       // epilogue warps (one per TMEM sub-partition)
constexpr int kPfDqWarps = 16;      // dequantising warps (four per TMEM sub-partition)
constexpr int kPfThreads = (2 + kPfEpWarps + kPfDqWarps + 1) * 32;   // + second MMA issuer (gate/up)
constexpr int kPfIssuer2Warp = 2 + kPfEpWarps + kPfDqWarps;
constexpr int kPfAStagesMax = 8;    // deepest TMEM A ring (barrier arrays)

struct PfChunk { int slot, row0, ntok, pad; };
struct PfTile { int chunk, mb, pad0, pad1; };

// ------------------------------------------------------------------ activations -> fp16, grouped order
// xh[r][8j + p] = x[pair_token[r]][8j + perm(p)], perm = 0,4,1,5,2,6,3,7 for
// int4 weights (the order the int4 unpacking produces) and the identity for int8.
__global__ void gather_x_f16_kernel(FwdArgs a, __half* xh, int rows) {
  const int per_row = a.d / 8;
  const bool perm = a.qtype == COLI_Q_INT4_G128;
  const long long n = (long long)rows * per_row;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i / per_row), c = (int)(i % per_row) * 8;
    const int tok = a.pair_token[r];
    float v[8];
    if ((unsigned)tok >= (unsigned)a.T) {   // a row no pair filled (a rejected expert id): zeros
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.f;
    } else if (a.xtype == COLI_X_BF16) {
      const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + (size_t)tok * a.d + c);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = __uint_as_float(w[j] << 16);
        v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    } else {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + (size_t)tok * a.d + c);
      const float4 f0 = p[0], f1 = p[1];
      v[0] = f0.x; v[1] = f0.y; v[2] = f0.z; v[3] = f0.w; v[4] = f1.x; v[5] = f1.y; v[6] = f1.z; v[7] = f1.w;
    }
    if (a.idot) {
      // integer-dot inputs: a block of 32 inputs is held by 4 consecutive lanes (d / 8 is a
      // multiple of 4 and so is every lane's index, so a group is inside or outside the loop
      // as a whole); the values q * 2^(e-6) are exact in fp16 for 2^-18 <= max |v| < 2^16
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
      const unsigned grp = 0xFu << (threadIdx.x & 28);
      m = fmaxf(m, __shfl_xor_sync(grp, m, 1));
      m = fmaxf(m, __shfl_xor_sync(grp, m, 2));
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = idot_value(v[j], m);
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = perm ? v[j] : v[2 * j], hi = perm ? v[j + 4] : v[2 * j + 1];
      o[j] = (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
    }
    *reinterpret_cast<uint4*>(xh + (size_t)r * a.d + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ------------------------------------------------------------------ chunk and tile tables
// One CTA: experts with tokens (ascending, shared last) are cut into chunks of
// up to kPfN tokens; every chunk yields one tile per 128 output rows.
__global__ void __launch_bounds__(256) plan_tiles_kernel(FwdArgs a, PfChunk* chunks, PfTile* gu_tiles,
                                                         PfTile* dn_tiles, int32_t* counts) {
  __shared__ int warp_tot[32];
  __shared__ int total;
  __shared__ int s_nchunks;
  const int tid = threadIdx.x;
  const int n_slots = a.n_unique[0] + (a.has_shared ? 1 : 0);
  // chunks
  int carry = 0;
  for (int b = 0; b < n_slots; b += 256) {
    const int i = b + tid;
    int slot = 0, pbeg = 0, cnt = 0, nch = 0;
    if (i < n_slots) {
      slot = a.unique[i];
      pbeg = a.offsets[slot];
      cnt = a.offsets[slot + 1] - pbeg;
      nch = (cnt + kPfN - 1) / kPfN;
    }
    const int ex = block_exclusive_scan(nch, warp_tot, &total);
    for (int c = 0; c < nch; ++c) {
      PfChunk ch;
      ch.slot = slot;
      ch.row0 = pbeg + c * kPfN;
      ch.ntok = min(kPfN, cnt - c * kPfN);
      ch.pad = 0;
      chunks[carry + ex + c] = ch;
    }
    carry += total;
  }
  if (tid == 0) s_nchunks = carry;
  __syncthreads();
  const int nch = s_nchunks;
  // tiles: every chunk has F / 128 gate/up tiles (F_shared / 128 for the shared
  // expert's chunks, which come last) and d / 128 down tiles; chunk-major order,
  // written by all threads at once
  const int n_sh = a.has_shared ? (a.T + kPfN - 1) / kPfN : 0;   // shared chunks (the last n_sh)
  const int n_rt = nch - n_sh;
  const int gm = a.F / kPfM, gms = a.Fs / kPfM, dm = a.d / kPfM;
  const int n_gu = n_rt * gm + n_sh * gms, n_dn = nch * dm;
  for (int i = tid; i < n_gu; i += blockDim.x) {
    int c, m;
    if (i < n_rt * gm) { c = i / gm; m = i - c * gm; }
    else { const int j = i - n_rt * gm; c = n_rt + j / gms; m = j - (j / gms) * gms; }
    gu_tiles[i] = PfTile{c, m, 0, 0};
  }
  for (int i = tid; i < n_dn; i += blockDim.x) {
    const int c = i / dm;
    dn_tiles[i] = PfTile{c, i - c * dm, 0, 0};
  }
  if (tid == 0) {
    counts[0] = nch;
    counts[1] = n_gu;
    counts[2] = n_dn;
  }
}

// ------------------------------------------------------------------ tcgen05 helpers (prefill)

// The eight K16 MMAs of one matrix and one K128 pipeline stage in one block:
// A = 64 TMEM columns, B = two 128-byte atoms 16 * atom16 bytes apart.  The
// issuing thread is on the critical path of the tensor pipe, so it executes as
// few instructions per MMA as possible.  `kb` = 0 for the tile's first stage
// (overwrite the accumulators), non-zero after (add to them).
__device__ __forceinline__ void umma_k128(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t kb,
                                              uint32_t atom16) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t.reg .b64 b1, b2, b3, b4, b5, b6, b7, bb;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, 0, 0;\n\t"
      "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\tadd.u32 a4, %1, 32;\n\t"
      "add.u32 a5, %1, 40;\n\tadd.u32 a6, %1, 48;\n\tadd.u32 a7, %1, 56;\n\t"
      "cvt.u64.u32 bb, %5;\n\t"
      "add.u64 b1, %2, 2;\n\tadd.u64 b2, %2, 4;\n\tadd.u64 b3, %2, 6;\n\t"
      "add.u64 b4, %2, bb;\n\tadd.u64 b5, b4, 2;\n\tadd.u64 b6, b4, 4;\n\tadd.u64 b7, b4, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %3, q;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(kb), "r"(atom16));
}

__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// fp16 pairs from the nibbles of a 32-bit word, exact, one logic op each:
// bits 0-3 / 16-19 -> 1024 + c (exponent 10: mantissa unit 1),
// bits 4-7 / 20-23 -> 64 + c   (exponent 6: mantissa bit 4 has weight 1).
__device__ __forceinline__ uint32_t nib_lo_h1024(uint32_t x) { return (x & 0x000F000Fu) | 0x64006400u; }
__device__ __forceinline__ uint32_t nib_hi_h64(uint32_t x) { return (x & 0x00F000F0u) | 0x54005400u; }

// Physical 16-byte chunk of logical chunk c in row r of a TMA box with rows of
// RB bytes stored with the RB-byte swizzle (RB = 32, 64 or 128).
template <int RB>
__device__ __forceinline__ int swz_chunk(int r, int c) {
  return c ^ (((r * RB) >> 7) & (RB / 16 - 1));
}

// ------------------------------------------------------------------ the grouped GEMM

struct PfArgs {
  const PfChunk* chunks;
  const PfTile* tiles;
  const int32_t* n_tiles;      // device scalar
  const CUtensorMap* wmaps;    // [(E+1)*3] raw-code maps (box: one stage of codes x 128 rows)
  __half* hout;                // gate/up: H [rows][Fmax] fp16 (column-permuted for int4)
  float* yout;                 // down: Y [rows][d] fp32
};

// TMEM: accumulators in columns [0, 2 * kPfN) (gate/up: gate and up of one
// tile; down: two tiles, double-buffered), then the ring of A stages
constexpr int kPfACol = 2 * kPfN;
static_assert(kPfN == 64 || kPfN == 128, "chunk size");

template <int QT, bool GU>
struct PfLayout {
  static constexpr int kMats = GU ? 2 : 1;
  static constexpr int kStageK = prefill_stage_k(GU);            // K per stage (64 or 128)
  static constexpr int kAtoms = kStageK / 64;                    // 128-byte activation atoms per stage
  static constexpr int kRawRow = prefill_raw_row_bytes(QT, GU);  // bytes of one row's codes per stage
  static constexpr int kRawBytes = kPfM * kRawRow;               // per matrix
  static constexpr int kBAtomBytes = kPfN * 128;                 // 128 token rows x 64 fp16
  static constexpr int kBBytes = kAtoms * kBAtomBytes;
  static constexpr int kStageBytes = kBBytes + kMats * kRawBytes;
  static constexpr int kStagesFit = (216 * 1024) / kStageBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static constexpr int kSmemBytes = kStages * kStageBytes;
  static constexpr int kAccSets = GU ? 1 : 2;                    // TMEM columns 0..255 hold the accumulators
  static constexpr int kTmaPerA = 1;                             // TMA stages per TMEM A stage
  static constexpr int kAStageCols = kMats * kStageK * kTmaPerA / 2;  // two fp16 per TMEM column
  static constexpr int kAStages = (512 - kPfACol) / kAStageCols;   // TMEM A ring depth
  static constexpr int kParts = kMats * kStageK / 32 / 4;        // 32-code parts per dequantising thread
  static_assert(kAStages <= kPfAStagesMax, "A ring");
  static constexpr int kCodesPerThread = 32;                     // per dequantising thread and stage
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(kRawRow == 32 || kRawRow == 64 || kRawRow == 128, "raw box width");
  static_assert(kAStages * kAStageCols + kPfACol <= 512, "TMEM budget");
};

// ID (gate/up only): integer-dot inputs, h leaves the epilogue as its IDOT values
template <int QT, bool GU, bool ID>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_ffn_kernel(FwdArgs a, PfArgs p, const __grid_constant__ CUtensorMap bmap) {
  using L = PfLayout<QT, GU>;
  constexpr bool I4 = QT == COLI_Q_INT4_G128;
  constexpr int S = L::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t tma_full[S], tma_empty[S], a_full[kPfAStagesMax], a_empty[kPfAStagesMax], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = *p.n_tiles;
  volatile int* abort_v = &abort_flag;

  if (threadIdx.x == 0) {
    constexpr int NI = GU ? 2 : 1;   // MMA-issuing threads (each commits)
    for (int s = 0; s < S; ++s) {
      mbar_init(&tma_full[s], 1);
      mbar_init(&tma_empty[s], NI);
    }
    for (int s = 0; s < L::kAStages; ++s) {
      mbar_init(&a_full[s], kPfDqWarps);
      mbar_init(&a_empty[s], NI);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], NI);
      mbar_init(&acc_empty[s], kPfEpWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  auto tile_info = [&](int t, int& slot, int& row0, int& ntok, int& mb, int& K) {
    const PfTile tl = p.tiles[t];
    const PfChunk ch = p.chunks[tl.chunk];
    slot = ch.slot;
    row0 = ch.row0;
    ntok = ch.ntok;
    mb = tl.mb;
    K = GU ? a.d : (slot == a.E ? a.Fs : a.F);
    if (a.slot_of) slot = __ldg(a.slot_of + slot);   // where the expert's weights are stored
  };
  auto fail_wait = [&]() {
    set_status(a.status, COLI_DEV_WAIT_TIMEOUT);
    atomicExch(&abort_flag, 1);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      // raw weight codes come from HBM: an L2 prefetch runs kPfPrefetch stages ahead of the
      // loads (also across tile boundaries) so that the loads into shared memory hit L2
      constexpr int kPfPrefetch = 8;
      int pf_t = blockIdx.x, pf_kb = 0, pf_nkb = 0, pf_slot = 0, pf_mb = 0;
      auto pf_load = [&]() {
        if (pf_t < n_tiles) {
          int r0, nt, K;
          tile_info(pf_t, pf_slot, r0, nt, pf_mb, K);
          pf_nkb = K / L::kStageK;
        }
      };
      auto pf_step = [&]() {
        if (pf_t >= n_tiles) return;
        for (int m = 0; m < L::kMats; ++m)
          tma_prefetch_2d(p.wmaps + (size_t)pf_slot * 3 + (GU ? m : 2), pf_kb * L::kRawRow, pf_mb * kPfM);
        if (++pf_kb == pf_nkb) { pf_kb = 0; pf_t += gridDim.x; pf_load(); }
      };
      pf_load();
      for (int j = 0; j < kPfPrefetch; ++j) pf_step();
      int it = 0;
      for (int t = blockIdx.x; t < n_tiles && !*abort_v; t += gridDim.x) {
        int slot, row0, ntok, mb, K;
        tile_info(t, slot, row0, ntok, mb, K);
        const int nkb = K / L::kStageK, nbox = (ntok + kPfBBox - 1) / kPfBBox;
        const uint32_t tx = (uint32_t)(L::kMats * L::kRawBytes + L::kAtoms * nbox * kPfBBox * 128);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          pf_step();
          const int s = it % S;
          if (it >= S && !mbar_wait(&tma_empty[s], ((it / S) - 1) & 1, a.wait_ns)) { ok = false; break; }
          uint8_t* st = smem + (size_t)s * L::kStageBytes;
          // failure-path test: CTA 0 withholds its first gate/up stage, so that every role waiting
          // on it reaches the (shortened) wait limit and the kernel stops with the status set
          if (GU && it == 0 && blockIdx.x == 0 && (a.inject & COLI_INJECT_WITHHOLD_STAGE)) continue;
          mbar_arrive_expect_tx(&tma_full[s], tx);
          for (int m = 0; m < L::kMats; ++m)
            tma_load_2d_nohint(st + L::kBBytes + m * L::kRawBytes, p.wmaps + (size_t)slot * 3 + (GU ? m : 2),
                               kb * L::kRawRow, mb * kPfM, &tma_full[s]);
          for (int at = 0; at < L::kAtoms; ++at)
            for (int b = 0; b < nbox; ++b)
              tma_load_2d_nohint(st + at * L::kBAtomBytes + b * kPfBBox * 128, &bmap, kb * L::kStageK + at * 64,
                                 row0 + b * kPfBBox, &tma_full[s]);
        }
        if (!ok) { fail_wait(); break; }
      }
      // drain: every issued stage must have landed before the CTA can exit
      const int issued = it;
      for (int j = (issued > S ? issued - S : 0); j < issued; ++j) mbar_wait(&tma_full[j % S], (j / S) & 1, a.wait_ns);
    }
  } else if (warp == 1 || (GU && warp == kPfIssuer2Warp)) {
    // ---------------------------------------------------------------- MMA issuers (gate/up: gate | up)
    const int mi = warp == 1 ? 0 : 1;
    if (lane == 0) {
      int it = 0, ia = 0, tcount = 0;   // TMA stages, TMEM A stages, tiles
      for (int t = blockIdx.x; t < n_tiles && !*abort_v; t += gridDim.x, ++tcount) {
        int slot, row0, ntok, mb, K;
        tile_info(t, slot, row0, ntok, mb, K);
        const int ntma = K / L::kStageK, nA = (ntma + L::kTmaPerA - 1) / L::kTmaPerA;
        const int N = (ntok + 15) & ~15;
        const uint32_t idesc = umma_idesc_f16(kPfM, N);
        const int acc = GU ? 0 : (tcount & 1);
        const int uses = GU ? tcount : (tcount >> 1);   // earlier tiles that used this accumulator set
        if (uses > 0) {
          if (!mbar_wait_spin(&acc_empty[acc], (uses - 1) & 1, a.wait_ns)) { fail_wait(); break; }
          tc_fence_after();
        }
        const uint32_t dacc = tmem + (uint32_t)(acc * kPfN);
        bool ok = true;
        for (int j = 0; j < nA; ++j, ++ia) {
          const int as = ia % L::kAStages;
          // a_full also covers the TMA data of the A stage's TMA stages: every dequantising warp
          // waited for their tma_full (raw codes and activations share that barrier) before arriving
          if (!mbar_wait_spin(&a_full[as], (ia / L::kAStages) & 1, a.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t A = tmem + (uint32_t)(kPfACol + as * L::kAStageCols);
          const int nsub = min(L::kTmaPerA, ntma - j * L::kTmaPerA);
          for (int sub = 0; sub < nsub; ++sub, ++it) {
            const int s = it % S;
            const uint64_t bd = umma_desc_sw128(smem_u32(smem + (size_t)s * L::kStageBytes));
            const uint32_t kbf = (j > 0 || sub > 0) ? 1u : 0u;   // 0: the tile's first MMAs overwrite
            if (GU) {
              umma_k128(dacc + mi * kPfN, A + mi * (L::kStageK / 2), bd, idesc, kbf,
                            (uint32_t)(L::kBAtomBytes >> 4));
            } else {
              umma_k128(dacc, A + sub * (L::kStageK / 2), bd, idesc, kbf, (uint32_t)(L::kBAtomBytes >> 4));
            }
            umma_commit(&tma_empty[s]);
          }
          umma_commit(&a_empty[as]);
        }
        if (!ok) { fail_wait(); break; }
        umma_commit(&acc_full[acc]);
      }
      // wait for the MMAs in flight before the CTA releases TMEM
      if (ia > 0) mbar_wait(&a_empty[(ia - 1) % L::kAStages], ((ia - 1) / L::kAStages) & 1, a.wait_ns);
    }
  } else if (warp < 2 + kPfEpWarps) {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int sp = warp & 3;                       // TMEM sub-partition: lanes 32*sp .. +31
    int tcount = 0;
    for (int t = blockIdx.x; t < n_tiles && !*abort_v; t += gridDim.x, ++tcount) {
      int slot, row0, ntok, mb, K;
      tile_info(t, slot, row0, ntok, mb, K);
      const int acc = GU ? 0 : (tcount & 1);
      const int uses = GU ? tcount : (tcount >> 1);
      if (!mbar_wait(&acc_full[acc], uses & 1, a.wait_ns)) { fail_wait(); break; }
      tc_fence_after();
      const DevExpert& ex = a.experts[slot];
      const int orow = mb * kPfM + sp * 32 + lane;  // weight row of this thread (TMEM lane)
      const uint32_t lane_addr = tmem + ((uint32_t)(sp * 32) << 16) + (uint32_t)(acc * kPfN);
      float s0 = 1.f, s1 = 1.f;
      if (!I4) {
        s0 = __ldg(static_cast<const float*>(ex.m[GU ? 0 : 2].s) + orow);
        if (GU) s1 = __ldg(static_cast<const float*>(ex.m[1].s) + orow);
      }
      // column of H that holds hidden unit orow (see the file header)
      const int hcol = I4 ? ((orow & ~7) | ((orow & 3) << 1) | ((orow >> 2) & 1)) : orow;
      const int ngroups = (ntok + 15) / 16;
      for (int g16 = 0; g16 < ngroups; ++g16) {
        uint32_t r0[16];
        tmem_ld16_issue(lane_addr + g16 * 16, r0);
        if (GU) {
          uint32_t r1[16];
          tmem_ld16_issue(lane_addr + kPfN + g16 * 16, r1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int tcol = g16 * 16 + i;
            if (tcol < ntok) {
              const float gv = __uint_as_float(r0[i]) * s0, uv = __uint_as_float(r1[i]) * s1;
              // SiLU with the fast exponential and division (relative error ~1e-6, far below the
              // fp16 rounding of h); the epilogue shares issue slots with the dequantising warps
              float hv = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
              if constexpr (ID) {   // the warp's 32 rows are one block of 32 hidden units; the block's
                                    // largest magnitude (non-negative floats order as their bits)
                const float m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv))));
                hv = idot_value(hv, m);
              }
              p.hout[(size_t)(row0 + tcol) * a.Fmax + hcol] = __float2half_rn(hv);
            }
          }
        } else {
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int tcol = g16 * 16 + i;
            if (tcol < ntok) p.yout[(size_t)(row0 + tcol) * a.d + orow] = __uint_as_float(r0[i]) * s0;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  } else if (warp < kPfIssuer2Warp) {
    // ---------------------------------------------------------------- dequantise (warps 6..21)
    // thread = (TMEM lane = weight row r, group g): per stage L::kParts parts of 32 codes of row r.
    // gate/up: g -> matrix g & 1, K quarters 2*(g >> 1) and +1; down: g -> K quarter g.
    const int sp = warp & 3, r = sp * 32 + lane;
    const int g = (warp - 2 - kPfEpWarps) >> 2;      // 0..3
    const int mat_i = GU ? (g & 1) : 0;
    const int kpart = GU ? (g >> 1) * L::kParts : g;  // first part
    const uint32_t tcol = (uint32_t)(mat_i * (L::kStageK / 2) + kpart * 16);
    const uint32_t tlane = (uint32_t)(sp * 32) << 16;
    int it = 0, ia = 0;   // TMA stages, TMEM A stages
    for (int t = blockIdx.x; t < n_tiles && !*abort_v; t += gridDim.x) {
      int slot, row0, ntok, mb, K;
      tile_info(t, slot, row0, ntok, mb, K);
      const int nkb = K / L::kStageK;
      const DevMat& M = a.experts[slot].m[GU ? mat_i : 2];
      const int wrow = mb * kPfM + r;
      const int G = K / 128, ZB = (G + 1) / 2;
      uint32_t zz8 = 0;
      if (!I4) zz8 = (0x6400u | (uint32_t)__ldg(M.z + wrow)) * 0x10001u;   // half2(1024 + z)
      // int4 scales / zero points: the row's 8-group batches (16 bytes of fp16 scales, 4 bytes
      // of zero nibbles) are loaded a batch ahead when the layout allows vector loads,
      // otherwise the stage's group is loaded one stage ahead
      const uint16_t* srow = static_cast<const uint16_t*>(M.s) + (size_t)wrow * G;
      const uint8_t* zrow = M.z + (size_t)wrow * ZB;
      const bool vec = I4 && (G & 7) == 0 && ((reinterpret_cast<uintptr_t>(M.s) & 15) == 0) &&
                       ((reinterpret_cast<uintptr_t>(M.z) & 3) == 0);
      const int nbatch = G / 8;
      uint4 sb = make_uint4(0, 0, 0, 0), sbn = sb;
      uint32_t zb = 0, zbn = 0;
      int cur_batch = 0;
      auto load_batch = [&](int b, uint4& sv, uint32_t& zv) {
        sv = __ldg(reinterpret_cast<const uint4*>(srow) + b);
        zv = __ldg(reinterpret_cast<const uint32_t*>(zrow) + b);
      };
      auto grp_of = [&](int kb) { return (kb * L::kStageK + kpart * 32) / 128; };
      auto load_sz = [&](int kb, uint32_t& sraw, uint32_t& zraw) {
        const int grp = grp_of(kb);
        sraw = __ldg(srow + grp);
        zraw = (__ldg(zrow + (grp >> 1)) >> ((grp & 1) * 4)) & 15u;
      };
      uint32_t s_next = 0, z_next = 0;
      if (vec) {
        load_batch(0, sb, zb);
        if (nbatch > 1) load_batch(1, sbn, zbn);
      } else if (I4) {
        load_sz(0, s_next, z_next);
      }
      bool ok = true;
      const int nA = (nkb + L::kTmaPerA - 1) / L::kTmaPerA;
      for (int j = 0; j < nA && ok; ++j, ++ia) {
        const int as = ia % L::kAStages;
        if (ia >= L::kAStages) {
          if (!mbar_wait(&a_empty[as], ((ia / L::kAStages) - 1) & 1, a.wait_ns)) { ok = false; break; }
          tc_fence_after();
        }
        const int nsub = min(L::kTmaPerA, nkb - j * L::kTmaPerA);
        for (int sub = 0; sub < nsub; ++sub, ++it) {
        const int kb = j * L::kTmaPerA + sub, s = it % S;
        uint32_t ss = 0, zz = zz8, zzh = 0;
        if (I4) {
          uint32_t sraw, zraw;
          if (vec) {
            const int grp = grp_of(kb);
            if ((grp >> 3) != cur_batch) {
              ++cur_batch;
              sb = sbn;
              zb = zbn;
              if (cur_batch + 1 < nbatch) load_batch(cur_batch + 1, sbn, zbn);
            }
            const int gi = grp & 7;
            const uint32_t sw = gi < 2 ? sb.x : gi < 4 ? sb.y : gi < 6 ? sb.z : sb.w;
            sraw = (sw >> ((gi & 1) * 16)) & 0xFFFFu;
            zraw = (zb >> (gi * 4)) & 15u;
          } else {
            sraw = s_next;
            zraw = z_next;
            if (kb + 1 < nkb) load_sz(kb + 1, s_next, z_next);
          }
          ss = sraw * 0x10001u;
          zz = (0x6400u | zraw) * 0x10001u;          // half2(1024 + z)
          zzh = (0x5400u | (zraw << 4)) * 0x10001u;  // half2(64 + z)
        }
        if (!mbar_wait(&tma_full[s], (it / S) & 1, a.wait_ns)) { ok = false; break; }
        const uint8_t* raw = smem + (size_t)s * L::kStageBytes + L::kBBytes + (GU ? mat_i * L::kRawBytes : 0) +
                             r * L::kRawRow;
#pragma unroll
        for (int pp = 0; pp < L::kParts; ++pp) {
          const int kp = kpart + pp;
          uint32_t o[16];
          if (I4) {
            const uint4 q = lds128(smem_u32(raw + (swz_chunk<L::kRawRow>(r, kp) << 4)));
            const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t q8 = qw[j] >> 8;
              o[4 * j + 0] = h2_mul(h2_sub(nib_lo_h1024(qw[j]), zz), ss);
              o[4 * j + 1] = h2_mul(h2_sub(nib_hi_h64(qw[j]), zzh), ss);
              o[4 * j + 2] = h2_mul(h2_sub(nib_lo_h1024(q8), zz), ss);
              o[4 * j + 3] = h2_mul(h2_sub(nib_hi_h64(q8), zzh), ss);
            }
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint4 q = lds128(smem_u32(raw + (swz_chunk<L::kRawRow>(r, 2 * kp + h) << 4)));
              const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                o[8 * h + 2 * j] = h2_sub(__byte_perm(qw[j], 0x64646464u, 0x4140), zz);
                o[8 * h + 2 * j + 1] = h2_sub(__byte_perm(qw[j], 0x64646464u, 0x4342), zz);
              }
            }
          }
          tmem_st16(tmem + tlane + (uint32_t)(kPfACol + as * L::kAStageCols + sub * (L::kStageK / 2)) + tcol +
                        pp * 16,
                    o);
        }
        }   // TMA stages of this A stage
        __syncwarp();
        tmem_st_wait();                 // also on the abort path: no store may be in flight at teardown
        if (!ok) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[as]);
      }
      if (!ok) { fail_wait(); break; }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
  }
}

// ------------------------------------------------------------------ host side

template <int QT, bool GU, bool ID = false>
static cudaError_t launch_pf(const FwdArgs& a, const PfArgs& p, const CUtensorMap& bmap, cudaStream_t st,
                             int num_sms) {
  using L = PfLayout<QT, GU>;
  const size_t smem = (size_t)L::kSmemBytes + 1024;
  static_assert(L::kSmemBytes + 1024 <= 227 * 1024, "shared memory");
  auto kern = prefill_ffn_kernel<QT, GU, ID>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms, kPfThreads, smem, st>>>(a, p, bmap);
  return cudaGetLastError();
}

cudaError_t launch_gather_x(const FwdArgs& a, __half* xh, int rows, cudaStream_t st) {
  const long long n = (long long)rows * (a.d / 8);
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  gather_x_f16_kernel<<<blocks, 256, 0, st>>>(a, xh, rows);
  return cudaGetLastError();
}

cudaError_t launch_plan_tiles(const FwdArgs& a, void* chunks, void* gu_tiles, void* dn_tiles, int32_t* counts,
                              cudaStream_t st) {
  plan_tiles_kernel<<<1, 256, 0, st>>>(a, static_cast<PfChunk*>(chunks), static_cast<PfTile*>(gu_tiles),
                                       static_cast<PfTile*>(dn_tiles), counts);
  return cudaGetLastError();
}

cudaError_t launch_prefill_gateup(const FwdArgs& a, const void* chunks, const void* tiles, const int32_t* n_tiles,
                                  const CUtensorMap* wmaps, const CUtensorMap& xmap, __half* hout, cudaStream_t st,
                                  int num_sms) {
  PfArgs p{static_cast<const PfChunk*>(chunks), static_cast<const PfTile*>(tiles), n_tiles, wmaps, hout, nullptr};
  if (a.idot)
    return a.qtype == COLI_Q_INT4_G128 ? launch_pf<COLI_Q_INT4_G128, true, true>(a, p, xmap, st, num_sms)
                                       : launch_pf<COLI_Q_INT8_PC, true, true>(a, p, xmap, st, num_sms);
  return a.qtype == COLI_Q_INT4_G128 ? launch_pf<COLI_Q_INT4_G128, true>(a, p, xmap, st, num_sms)
                                     : launch_pf<COLI_Q_INT8_PC, true>(a, p, xmap, st, num_sms);
}

cudaError_t launch_prefill_down(const FwdArgs& a, const void* chunks, const void* tiles, const int32_t* n_tiles,
                                const CUtensorMap* wmaps, const CUtensorMap& hmap, float* yout, cudaStream_t st,
                                int num_sms) {
  PfArgs p{static_cast<const PfChunk*>(chunks), static_cast<const PfTile*>(tiles), n_tiles, wmaps, nullptr, yout};
  return a.qtype == COLI_Q_INT4_G128 ? launch_pf<COLI_Q_INT4_G128, false>(a, p, hmap, st, num_sms)
                                     : launch_pf<COLI_Q_INT8_PC, false>(a, p, hmap, st, num_sms);
}

}  // namespace coli
