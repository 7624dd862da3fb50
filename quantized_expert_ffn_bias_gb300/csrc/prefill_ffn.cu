// Expert FFN for large token counts (prefill, batched verification): grouped
// GEMMs on the 5th-generation tensor cores (tcgen05, accumulators in TMEM).
//
// Each chosen expert's weights are dequantised once per chunk of up to 256 of
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
// CTA (persistent, one per SM): warp 0 issues TMA loads (raw codes, activation
// rows), warp 1 owns TMEM and issues the MMAs (one thread), warps 2..9
// dequantise into 128-byte-swizzled K-major tiles and run the epilogue.  All
// waits are bounded; a timeout sets the status word and every role stops.
#include "moe_internal.cuh"

namespace coli {

constexpr int kPfM = 128;          // weight rows per tile (MMA M)
constexpr int kPfN = 256;          // tokens per chunk (largest MMA N)
constexpr int kPfKB = 64;          // K elements per stage (one 128-byte swizzle atom of fp16)
constexpr int kPfBBox = 64;        // activation rows per TMA box
constexpr int kPfDqWarps = 8;
constexpr int kPfThreads = (2 + kPfDqWarps) * 32;
constexpr int kPfABytes = kPfM * 128;      // 16 KB per matrix
constexpr int kPfBBytes = kPfN * 128;      // 32 KB

struct PfChunk { int slot, row0, ntok, pad; };
struct PfTile { int chunk, mb, pad0, pad1; };

// ------------------------------------------------------------------ activations -> fp16, grouped order
__global__ void gather_x_f16_kernel(FwdArgs a, __half* xh, int rows) {
  const int per_row = a.d / 8;
  const long long n = (long long)rows * per_row;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i / per_row), c = (int)(i % per_row) * 8;
    const int tok = a.pair_token[r];
    float v[8];
    if (a.xtype == COLI_X_BF16) {
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
    uint4 o;
    o.x = __half_as_ushort(__float2half_rn(v[0])) | ((uint32_t)__half_as_ushort(__float2half_rn(v[1])) << 16);
    o.y = __half_as_ushort(__float2half_rn(v[2])) | ((uint32_t)__half_as_ushort(__float2half_rn(v[3])) << 16);
    o.z = __half_as_ushort(__float2half_rn(v[4])) | ((uint32_t)__half_as_ushort(__float2half_rn(v[5])) << 16);
    o.w = __half_as_ushort(__float2half_rn(v[6])) | ((uint32_t)__half_as_ushort(__float2half_rn(v[7])) << 16);
    *reinterpret_cast<uint4*>(xh + (size_t)r * a.d + c) = o;
  }
}

// ------------------------------------------------------------------ chunk and tile tables
// One CTA: experts with tokens (ascending, shared last) are cut into chunks of
// up to 256 tokens; every chunk yields one tile per 128 output rows.
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
  // tiles: gate/up rows F (F_shared for the shared slot), down rows d
  int gcarry = 0, dcarry = 0;
  for (int b = 0; b < nch; b += 256) {
    const int c = b + tid;
    int gm = 0, dm = 0;
    if (c < nch) {
      const int slot = chunks[c].slot;
      gm = (slot == a.E ? a.Fs : a.F) / kPfM;
      dm = a.d / kPfM;
    }
    const int gex = block_exclusive_scan(gm, warp_tot, &total);
    const int gtot = total;
    const int dex = block_exclusive_scan(dm, warp_tot, &total);
    const int dtot = total;
    for (int m = 0; m < gm; ++m) gu_tiles[gcarry + gex + m] = PfTile{c, m, 0, 0};
    for (int m = 0; m < dm; ++m) dn_tiles[dcarry + dex + m] = PfTile{c, m, 0, 0};
    gcarry += gtot;
    dcarry += dtot;
  }
  if (tid == 0) {
    counts[0] = nch;
    counts[1] = gcarry;
    counts[2] = dcarry;
  }
}

// ------------------------------------------------------------------ tcgen05 helpers

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

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
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

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 2D TMA load without cache hint (activation rows: reused across the m-blocks of a chunk).
__device__ __forceinline__ void tma_load_2d_nohint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// int4 -> fp16 pairs (1024 + code) in input order, see the file header
__device__ __forceinline__ void int4_word_to_h1024(uint32_t q, uint32_t (&h)[4]) {
  const uint32_t r = q >> 4;
  const uint32_t v0 = __byte_perm(q, r, 0x5410);
  const uint32_t v1 = __byte_perm(q, r, 0x7632);
  h[0] = (v0 & 0x000F000Fu) | 0x64006400u;
  h[1] = ((v0 >> 8) & 0x000F000Fu) | 0x64006400u;
  h[2] = (v1 & 0x000F000Fu) | 0x64006400u;
  h[3] = ((v1 >> 8) & 0x000F000Fu) | 0x64006400u;
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

// ------------------------------------------------------------------ the grouped GEMM

struct PfArgs {
  const PfChunk* chunks;
  const PfTile* tiles;
  const int32_t* n_tiles;      // device scalar
  const CUtensorMap* wmaps;    // [(E+1)*3] raw-code maps (box: 64 codes x 128 rows)
  __half* hout;                // gate/up: H [rows][Fmax] fp16
  float* yout;                 // down: Y [rows][d] fp32
};

template <int QT, bool GU>
struct PfLayout {
  static constexpr int kMats = GU ? 2 : 1;
  static constexpr int kRawRow = QT == COLI_Q_INT4_G128 ? 32 : 64;   // bytes of 64 codes
  static constexpr int kRawBytes = kPfM * kRawRow;
  static constexpr int kStageBytes = kMats * (kPfABytes + kRawBytes) + kPfBBytes;
  static constexpr int kStages = (220 * 1024) / kStageBytes;
  // stage: [A_0][A_1][B][raw_0][raw_1]  (A, B 1024-aligned)
  static constexpr int kOffB = kMats * kPfABytes;
  static constexpr int kOffRaw = kOffB + kPfBBytes;
  static constexpr int kTmemCols = GU ? 512 : 256;
};

template <int QT, bool GU>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_ffn_kernel(FwdArgs a, PfArgs p, const __grid_constant__ CUtensorMap bmap) {
  using L = PfLayout<QT, GU>;
  constexpr bool I4 = QT == COLI_Q_INT4_G128;
  constexpr int S = L::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t full_tma[S], full_a[S], empty[S], acc_full, acc_empty;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = *p.n_tiles;
  volatile int* abort_v = &abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_tma[s], 1);
      mbar_init(&full_a[s], kPfDqWarps);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, kPfDqWarps);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(L::kTmemCols));
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
  };
  auto fail_wait = [&]() {
    set_status(a.status, COLI_DEV_WAIT_TIMEOUT);
    atomicExch(&abort_flag, 1);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int it = 0;
      for (int t = blockIdx.x; t < n_tiles && !*abort_v; t += gridDim.x) {
        int slot, row0, ntok, mb, K;
        tile_info(t, slot, row0, ntok, mb, K);
        const int nkb = K / kPfKB, nbox = (ntok + kPfBBox - 1) / kPfBBox;
        const uint32_t tx = (uint32_t)(L::kMats * L::kRawBytes + nbox * kPfBBox * 128);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % S;
          if (it >= S && !mbar_wait(&empty[s], ((it / S) - 1) & 1)) { fail_wait(); break; }
          uint8_t* st = smem + (size_t)s * L::kStageBytes;
          mbar_arrive_expect_tx(&full_tma[s], tx);
          for (int m = 0; m < L::kMats; ++m)
            tma_load_2d_nohint(st + L::kOffRaw + m * L::kRawBytes, p.wmaps + (size_t)slot * 3 + (GU ? m : 2),
                               kb * L::kRawRow, mb * kPfM, &full_tma[s]);
          for (int b = 0; b < nbox; ++b)
            tma_load_2d_nohint(st + L::kOffB + b * kPfBBox * 128, &bmap, kb * kPfKB, row0 + b * kPfBBox,
                               &full_tma[s]);
        }
      }
      // drain: every issued stage must have landed before the CTA can exit
      const int issued = it;
      for (int j = (issued > S ? issued - S : 0); j < issued; ++j) mbar_wait(&full_tma[j % S], (j / S) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int it = 0, tcount = 0;
      for (int t = blockIdx.x; t < n_tiles && !*abort_v; t += gridDim.x, ++tcount) {
        int slot, row0, ntok, mb, K;
        tile_info(t, slot, row0, ntok, mb, K);
        const int nkb = K / kPfKB;
        const int N = (ntok + 15) & ~15;
        const uint32_t idesc = umma_idesc_f16(kPfM, N);
        if (tcount > 0) {
          if (!mbar_wait(&acc_empty, (tcount - 1) & 1)) { fail_wait(); break; }
          tc_fence_after();
        }
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % S;
          if (!mbar_wait(&full_a[s], (it / S) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + (size_t)s * L::kStageBytes);
#pragma unroll
          for (int k = 0; k < kPfKB / 16; ++k) {
            const uint64_t bd = umma_desc_sw128(st + L::kOffB + k * 32);
            for (int m = 0; m < L::kMats; ++m)
              umma_f16(tmem + m * 256, umma_desc_sw128(st + m * kPfABytes + k * 32), bd, idesc,
                       (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&empty[s]);
        }
        if (!ok) { fail_wait(); break; }
        umma_commit(&acc_full);
      }
      // wait for the MMAs in flight before the CTA releases TMEM
      if (it > 0) mbar_wait(&empty[(it - 1) % S], ((it - 1) / S) & 1);
    }
  } else {
    // ---------------------------------------------------------------- dequantise + epilogue (warps 2..9)
    const int dt = threadIdx.x - 64;               // 0..255
    const int r = dt & 127;                        // weight row within the tile
    const int half = dt >> 7;                      // gate/up: matrix; down: which 32 codes
    const int sp = warp & 3;                       // TMEM sub-partition of this warp
    const int colhalf = (warp - 2) >> 2;           // epilogue: which half of the 16-column groups
    int it = 0, tcount = 0;
    for (int t = blockIdx.x; t < n_tiles && !*abort_v; t += gridDim.x, ++tcount) {
      int slot, row0, ntok, mb, K;
      tile_info(t, slot, row0, ntok, mb, K);
      const int nkb = K / kPfKB;
      const DevExpert& ex = a.experts[slot];
      const int mat = GU ? half : 2;
      const DevMat& M = ex.m[mat];
      const int wrow = mb * kPfM + r;
      const int G = K / 128, ZB = (G + 1) / 2;
      uint32_t zz8 = 0;
      if (!I4) {
        const uint32_t z = __ldg(M.z + wrow);
        zz8 = (0x6400u | z) * 0x10001u;            // half2(1024 + z, 1024 + z)
      }
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int s = it % S;
        uint32_t ss = 0, zz = zz8;
        if (I4) {
          const int g = (kb * kPfKB) / 128;
          const uint16_t sb = __ldg(static_cast<const uint16_t*>(M.s) + (size_t)wrow * G + g);
          const uint32_t zb = __ldg(M.z + (size_t)wrow * ZB + (g >> 1));
          const uint32_t z = (zb >> ((g & 1) * 4)) & 15u;
          ss = (uint32_t)sb * 0x10001u;
          zz = (0x6400u | z) * 0x10001u;
        }
        if (!mbar_wait(&full_tma[s], (it / S) & 1)) { ok = false; break; }
        uint8_t* st = smem + (size_t)s * L::kStageBytes;
        uint8_t* A = st + (GU ? half * kPfABytes : 0);
        const uint8_t* raw = st + L::kOffRaw + (GU ? half * L::kRawBytes : 0) + r * L::kRawRow;
        // output 16-byte chunks c (8 fp16 each) of row r; down: this thread does 4 of the 8
        const int c0 = GU ? 0 : half * 4, nc = GU ? 8 : 4;
        for (int c = c0; c < c0 + nc; c += 4) {
          uint4 out[4];
          if (I4) {
            const uint4 q = *reinterpret_cast<const uint4*>(raw + c * 4);   // 32 codes
            const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t h[4];
              int4_word_to_h1024(qw[j], h);
              out[j].x = h2_mul(h2_sub(h[0], zz), ss);
              out[j].y = h2_mul(h2_sub(h[1], zz), ss);
              out[j].z = h2_mul(h2_sub(h[2], zz), ss);
              out[j].w = h2_mul(h2_sub(h[3], zz), ss);
            }
          } else {
            const uint4* q4 = reinterpret_cast<const uint4*>(raw + c * 8);  // 32 codes
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const uint4 q = q4[j];
              const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                uint32_t* o = reinterpret_cast<uint32_t*>(&out[2 * j + i]);
                o[0] = h2_sub(__byte_perm(qw[2 * i], 0x64646464u, 0x4140), zz);
                o[1] = h2_sub(__byte_perm(qw[2 * i], 0x64646464u, 0x4342), zz);
                o[2] = h2_sub(__byte_perm(qw[2 * i + 1], 0x64646464u, 0x4140), zz);
                o[3] = h2_sub(__byte_perm(qw[2 * i + 1], 0x64646464u, 0x4342), zz);
              }
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(A + r * 128 + (((c + j) ^ (r & 7)) << 4)) = out[j];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_a[s]);
      }
      if (!ok) { fail_wait(); break; }
      // ---- epilogue: wait for the tile's accumulators
      if (!mbar_wait(&acc_full, tcount & 1)) { fail_wait(); break; }
      tc_fence_after();
      const int trow = sp * 32 + lane;             // TMEM lane = weight row of this thread
      const int orow = mb * kPfM + trow;
      const uint32_t lane_addr = tmem + ((uint32_t)(sp * 32) << 16);
      float s0 = 1.f, s1 = 1.f;
      if (!I4) {
        s0 = __ldg(static_cast<const float*>(ex.m[GU ? 0 : 2].s) + orow);
        if (GU) s1 = __ldg(static_cast<const float*>(ex.m[1].s) + orow);
      }
      const int ngroups = (ntok + 15) / 16;
      for (int g16 = colhalf; g16 < ngroups; g16 += 2) {
        float v0[16];
        tmem_ld16(lane_addr + g16 * 16, v0);
        if (GU) {
          float v1[16];
          tmem_ld16(lane_addr + 256 + g16 * 16, v1);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int tcol = g16 * 16 + i;
            if (tcol < ntok) {
              const float gv = v0[i] * s0, uv = v1[i] * s1;
              const float hv = gv / (1.0f + expf(-gv)) * uv;
              p.hout[(size_t)(row0 + tcol) * a.Fmax + orow] = __float2half_rn(hv);
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int tcol = g16 * 16 + i;
            if (tcol < ntok) p.yout[(size_t)(row0 + tcol) * a.d + orow] = v0[i] * s0;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(L::kTmemCols));
  }
}

// ------------------------------------------------------------------ host side

template <int QT, bool GU>
static cudaError_t launch_pf(const FwdArgs& a, const PfArgs& p, const CUtensorMap& bmap, cudaStream_t st,
                             int num_sms) {
  using L = PfLayout<QT, GU>;
  const size_t smem = (size_t)L::kStages * L::kStageBytes + 1024;
  auto kern = prefill_ffn_kernel<QT, GU>;
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
