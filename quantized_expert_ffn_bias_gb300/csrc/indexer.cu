// Key selection of sparse attention: the "lightning indexer" scores and its
// top-k ("25GB RAM runs 744B GLM-5.2" page (pwwt.cn), section 3.3: every layer
// keeps the top-2048 causal keys; section 4.4: a light indexer scores the
// earlier keys and the top-k entries are selected, the indexer itself doing
// the scoring and the top-k).  The scoring formula is that of the DeepSeek-V3.2
// indexer the page cites:
//   I[t][s] = sum_{j < H} w[t][j] * relu(q[t][j] . k[s])
// for the keys s <= pos0 + t the query at position pos0 + t sees.
//
// Scores: a dense contraction of the keys [L][128] with the queries' heads
// [64 T][128] on the 5th-generation tensor cores (bf16 operands staged by TMA
// in shared memory, fp32 accumulators in tensor memory), one CTA per SM over
// tiles of 128 keys.  Warp 0 loads, warp 1 issues the MMAs (M = 128 keys,
// N = 64 heads x up to 4 queries, K = 128 in eight steps), warps 2..5 read the
// accumulators back and form relu, the head-weighted sum (heads in ascending
// order) and the causal mask.  Double-buffered accumulators let the MMAs of one
// tile overlap the epilogue of the previous one.  All waits are bounded.
//
// Top-k: one thread-block cluster of 8 CTAs per query runs an exact bucket
// select on the scores' order-preserving integer images held in shared
// memory, with the cluster's counts summed through distributed shared memory
// (see the selection kernel).
#include "moe_internal.cuh"

namespace coli {

constexpr int kIxKeys = 128;        // keys per tile (MMA M, TMEM lanes)
constexpr int kIxD = 128;           // head dimension (two 64-element swizzle atoms)
constexpr int kIxHeads = 64;        // heads per query
constexpr int kIxQMax = 4;          // queries per launch (MMA N = 64 * queries <= 256)
constexpr int kIxStages = 4;
constexpr int kIxThreads = 6 * 32;
constexpr int kIxAtomKeys = kIxKeys * 128;            // bytes of one 64-element atom of a key tile
constexpr int kIxStageBytes = 2 * kIxAtomKeys;        // 32 KB

struct IxArgs {
  int T, L, pos0;
  const float* w;        // [T][64] head weights of this launch's queries
  float* scores;         // [T][ls]
  int ls;
  int32_t* status;
  unsigned long long wait_ns;
};

// Order-preserving integer image of an fp32 value.
__device__ __forceinline__ uint32_t ix_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ix_unkey(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}



__global__ void __launch_bounds__(kIxThreads, 1)
    indexer_scores_kernel(IxArgs p, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t full[kIxStages], empty[kIxStages], q_full, acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base;
  __shared__ float ws[kIxQMax * kIxHeads];
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qs = smem + kIxStages * kIxStageBytes;   // queries: two atoms of N rows x 128 bytes
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = kIxHeads * p.T;
  const int n_tiles = (p.L + kIxKeys - 1) / kIxKeys;
  volatile int* abort_v = &abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kIxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 4);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < p.T * kIxHeads; i += blockDim.x) ws[i] = p.w[i];
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;
  auto fail_wait = [&]() {
    set_status(p.status, COLI_DEV_WAIT_TIMEOUT);
    atomicExch(&abort_flag, 1);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      mbar_arrive_expect_tx(&q_full, (uint32_t)(2 * N * 128));
      for (int at = 0; at < 2; ++at) tma_load_2d_nohint(qs + at * N * 128, &qmap, at * 64, 0, &q_full);
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles && !*abort_v; t += gridDim.x, ++it) {
        const int s = it % kIxStages;
        if (it >= kIxStages && !mbar_wait(&empty[s], ((it / kIxStages) - 1) & 1, p.wait_ns)) { ok = false; break; }
        uint8_t* st = smem + (size_t)s * kIxStageBytes;
        mbar_arrive_expect_tx(&full[s], (uint32_t)kIxStageBytes);
        for (int at = 0; at < 2; ++at) tma_load_2d_nohint(st + at * kIxAtomKeys, &kmap, at * 64, t * kIxKeys, &full[s]);
      }
      if (!ok) fail_wait();
      // drain: every issued copy lands before the CTA exits
      mbar_wait(&q_full, 0, p.wait_ns);
      for (int j = (it > kIxStages ? it - kIxStages : 0); j < it; ++j)
        mbar_wait(&full[j % kIxStages], (j / kIxStages) & 1, p.wait_ns);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kIxKeys, N);
      bool ok = mbar_wait_spin(&q_full, 0, p.wait_ns);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint64_t qd = umma_desc_sw128(smem_u32(qs));
      const uint64_t q_atom = (uint64_t)((N * 128) >> 4);
      int i = 0;
      for (int t = blockIdx.x; ok && t < n_tiles && !*abort_v; t += gridDim.x, ++i) {
        const int s = i % kIxStages, acc = i & 1;
        if (!mbar_wait_spin(&full[s], (i / kIxStages) & 1, p.wait_ns)) { ok = false; break; }
        if (i >= 2 && !mbar_wait_spin(&acc_empty[acc], ((i >> 1) - 1) & 1, p.wait_ns)) { ok = false; break; }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint64_t kd = umma_desc_sw128(smem_u32(smem + (size_t)s * kIxStageBytes));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // step kk: 16 elements (32 bytes) of atom kk / 4 of both operands
          const uint64_t off = (uint64_t)((kk & 3) * 2);
          const uint64_t a = kd + off + (kk >= 4 ? (uint64_t)(kIxAtomKeys >> 4) : 0);
          const uint64_t b = qd + off + (kk >= 4 ? q_atom : 0);
          umma_ss(tmem + (uint32_t)(acc * N), a, b, idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(&empty[s]);
        umma_commit(&acc_full[acc]);
      }
      if (!ok) fail_wait();
      // the last accumulators must be complete before the CTA frees tensor memory
      if (i > 0) mbar_wait(&acc_full[(i - 1) & 1], ((i - 1) >> 1) & 1, p.wait_ns);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int sp = warp & 3;                  // TMEM sub-partition: lanes 32 sp .. 32 sp + 31
    int i = 0;
    for (int t = blockIdx.x; t < n_tiles && !*abort_v; t += gridDim.x, ++i) {
      const int acc = i & 1;
      if (!mbar_wait(&acc_full[acc], (i >> 1) & 1, p.wait_ns)) { fail_wait(); break; }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int s = t * kIxKeys + sp * 32 + lane;
      const uint32_t taddr = tmem + ((uint32_t)(sp * 32) << 16) + (uint32_t)(acc * N);
      for (int q = 0; q < p.T; ++q) {
        // the query's 64 head columns: four 16-column loads in flight, one wait
        uint32_t r[kIxHeads / 16][16];
#pragma unroll
        for (int c = 0; c < kIxHeads / 16; ++c) tmem_ld16_issue(taddr + (uint32_t)(q * kIxHeads + c * 16), r[c]);
        tmem_ld_wait();
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < kIxHeads; ++j)
          sum = fmaf(ws[q * kIxHeads + j], fmaxf(__uint_as_float(r[j >> 4][j & 15]), 0.f), sum);
        const bool vis = s < p.L && s <= p.pos0 + q;
        if (s < p.L) p.scores[(size_t)q * p.ls + s] = vis ? sum : -INFINITY;
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
  }
}

// ------------------------------------------------------------------ top-k: one cluster of CTAs per query
//
// kIxSelCtas CTAs (one thread-block cluster) share a query's visible keys in contiguous ranges and keep
// their keys' integer images in shared memory.  An exact bucket select runs over the cluster: the
// cluster's smallest and largest image bound the range; each round every CTA counts its keys of the
// current range in 2048 bins (round 0 linear in the score value, later rounds in the image), the CTAs
// sum the cluster's counts through distributed shared memory, and the keys of the bin holding the
// topk-th largest key become the next range; within four rounds the range is one value.  Keys above
// that value are taken, and keys equal to it
// in ascending key order until topk keys are taken (a tie goes to the lower key).  A cluster prefix of
// the CTAs' counts places each CTA's keys in the ascending output.  Cluster barriers are hardware
// barriers; no CTA leaves while another may still read its shared memory.

constexpr int kIxSelCtas = 8;            // CTAs per query (portable cluster size)
constexpr int kIxSelThreads = 512;
constexpr int kIxBins = 2048;
constexpr int kIxGroups = kIxBins / 32;  // group sums exchanged first (a group: 32 bins)

struct IxSel {
  const float* scores;     // [T][ls]
  int ls, L, pos0, topk;
  int chunk;               // keys per CTA (a multiple of 32)
  int32_t* out;            // [T][topk]
  int32_t* status;
};

__device__ __forceinline__ void ix_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Generic address of shared variable `p` in CTA `rank` of this cluster.  Loads through it are ordinary
// loads: the compiler may batch them, and the cluster barrier (a memory clobber) orders them after it.
template <typename T>
__device__ __forceinline__ const T* ix_peer(const T* p, uint32_t rank) {
  uint64_t a;
  asm("mapa.u64 %0, %1, %2;" : "=l"(a) : "l"(reinterpret_cast<uint64_t>(p)), "r"(rank));
  return reinterpret_cast<const T*>(a);
}

__global__ void __launch_bounds__(kIxSelThreads, 1) indexer_select_kernel(IxSel p) {
  // per round and bin: keys, smallest and largest image (ping-pong: a peer may still read the previous
  // round's), then this CTA's keys' integer images
  extern __shared__ __align__(16) uint32_t dyn[];
  uint32_t(*cnt)[kIxBins] = reinterpret_cast<uint32_t(*)[kIxBins]>(dyn);
  uint32_t(*bmin)[kIxBins] = reinterpret_cast<uint32_t(*)[kIxBins]>(dyn + 2 * kIxBins);
  uint32_t(*bmax)[kIxBins] = reinterpret_cast<uint32_t(*)[kIxBins]>(dyn + 4 * kIxBins);
  uint32_t* u_s = dyn + 6 * kIxBins;
  __shared__ uint32_t ex[4];                            // exchanged: min image, max image, keys above, keys equal
  __shared__ uint32_t gsum[2][kIxGroups], gtot[kIxGroups];
  __shared__ uint32_t s_lo, s_hi;
  __shared__ int s_rem;
  __shared__ int warp_tot[32];
  __shared__ uint32_t wmin[32], wmax[32];
  __shared__ int total;
  const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, wid = tid >> 5, nw = nthr >> 5;
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int q = blockIdx.y;
  const long long v = (long long)p.pos0 + q + 1;          // keys s <= pos0 + q, s < L
  const int vis = v < p.L ? (int)v : p.L;
  const int topk = p.topk;
  int32_t* o = p.out + (size_t)q * topk;
  if (vis <= topk) {                                      // cluster-uniform: every visible key, then -1
    for (int i = (int)rank * nthr + tid; i < topk; i += kIxSelCtas * nthr) o[i] = i < vis ? i : -1;
    return;
  }
  const int k0 = (int)rank * p.chunk;
  const int n = max(0, min(vis, k0 + p.chunk) - k0);
  const float* sc = p.scores + (size_t)q * p.ls + k0;

  // load the images; the CTA's smallest and largest, then the cluster's; clear round 0's bins
  for (int b = tid; b < kIxBins; b += nthr) {
    cnt[0][b] = 0u;
    bmin[0][b] = 0xFFFFFFFFu;
    bmax[0][b] = 0u;
  }
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll 4
  for (int i = tid; i < n; i += nthr) {
    const uint32_t u = ix_key(__ldcg(sc + i));
    u_s[i] = u;
    mn = min(mn, u);
    mx = max(mx, u);
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) {
    wmin[wid] = mn;
    wmax[wid] = mx;
  }
  __syncthreads();
  if (wid == 0) {
    mn = __reduce_min_sync(0xffffffffu, lane < nw ? wmin[lane] : 0xFFFFFFFFu);
    mx = __reduce_max_sync(0xffffffffu, lane < nw ? wmax[lane] : 0u);
    if (lane == 0) {
      ex[0] = mn;
      ex[1] = mx;
    }
  }
  ix_cluster_sync();                                      // (1) every CTA's bounds are visible
  if (wid == 0) {
    mn = __reduce_min_sync(0xffffffffu, lane < kIxSelCtas ? *ix_peer(&ex[0], lane) : 0xFFFFFFFFu);
    mx = __reduce_max_sync(0xffffffffu, lane < kIxSelCtas ? *ix_peer(&ex[1], lane) : 0u);
    if (lane == 0) {
      s_lo = mn;
      s_hi = mx;
    }
  }
  __syncthreads();

  // rounds: the keys with images in [lo, hi] hold the wanted key at rank `rem` from the top; 2048 bins over
  // the range (round 0 linear in the score value, then linear in the image), counted per CTA, summed over
  // the cluster; the bin holding rank `rem` becomes the range, bounded by its keys' smallest and largest
  // images.  The range shrinks by at least 2048 per image round, so it ends at one value.
  uint32_t lo = s_lo, hi = s_hi;
  int rem = topk;
  constexpr int kMaxRounds = 8;                          // 4 suffice (one value round, three image rounds)
  for (int round = 0; lo < hi && round < kMaxRounds; ++round) {
    const int pb = round & 1;
    const float vlo = ix_unkey(lo), vhi = ix_unkey(hi);
    const float vscale = (float)kIxBins / (vhi - vlo);
    const bool by_value = round == 0 && vscale > 0.f && vscale < INFINITY;
    const uint32_t width = (uint32_t)((((uint64_t)hi - lo) >> 11) + 1);
    for (int i = tid; i < n; i += nthr) {                 // (this round's bins were cleared before)
      const uint32_t u = u_s[i];
      if (u < lo || u > hi) continue;
      int b;
      if (by_value) {
        b = (int)((ix_unkey(u) - vlo) * vscale);
        b = b < 0 ? 0 : (b > kIxBins - 1 ? kIxBins - 1 : b);
      } else {
        b = (int)((u - lo) / width);
      }
      atomicAdd(&cnt[pb][b], 1u);
      atomicMin(&bmin[pb][b], u);
      atomicMax(&bmax[pb][b], u);
    }
    __syncthreads();
    // this CTA's group sums (64 groups of 32 bins), read by the peers: 4 bins a thread, 8 threads a group
    {
      static_assert(kIxBins == 4 * kIxSelThreads, "four bins per thread");
      const uint4 c4 = reinterpret_cast<const uint4*>(cnt[pb])[tid];
      uint32_t g = (c4.x + c4.y) + (c4.z + c4.w);
      g += __shfl_xor_sync(0xffffffffu, g, 1);
      g += __shfl_xor_sync(0xffffffffu, g, 2);
      g += __shfl_xor_sync(0xffffffffu, g, 4);
      if ((tid & 7) == 0) gsum[pb][tid >> 3] = g;
    }
    ix_cluster_sync();                                    // the round's counts are complete in every CTA
    // clear the next round's bins: every peer has finished reading them (it passed this barrier after
    // the round that last used them)
    for (int b = tid; b < kIxBins; b += nthr) {
      cnt[pb ^ 1][b] = 0u;
      bmin[pb ^ 1][b] = 0xFFFFFFFFu;
      bmax[pb ^ 1][b] = 0u;
    }
    // the group holding rank `rem` (counted from the top), from the cluster's group sums
    if (tid < kIxGroups) {
      const int g = kIxGroups - 1 - tid;                  // thread 0: the top group
      uint32_t part[kIxSelCtas];
#pragma unroll
      for (int r = 0; r < kIxSelCtas; ++r) part[r] = ix_peer(&gsum[pb][0], r)[g];
      uint32_t t = 0;
#pragma unroll
      for (int r = 0; r < kIxSelCtas; ++r) t += part[r];
      gtot[tid] = t;
    }
    __syncthreads();
    if (wid == 0) {
      // lanes own groups 2 lane and 2 lane + 1 from the top; prefix from the top
      const int t0 = (int)gtot[2 * lane], t1 = (int)gtot[2 * lane + 1];
      int inc = t0 + t1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v2 = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v2;
      }
      const int above = inc - t0 - t1;
      int gsel = -1, grem = 0;
      if (above < rem && rem <= above + t0) {
        gsel = kIxGroups - 1 - 2 * lane;
        grem = rem - above;
      } else if (above + t0 < rem && rem <= above + t0 + t1) {
        gsel = kIxGroups - 2 - 2 * lane;
        grem = rem - above - t0;
      }
      const unsigned who = __ballot_sync(0xffffffffu, gsel >= 0);
      const int src = who ? __ffs(who) - 1 : 0;
      gsel = __shfl_sync(0xffffffffu, gsel, src);
      grem = __shfl_sync(0xffffffffu, grem, src);
      if (gsel < 0) gsel = 0;                             // (not reached: the range holds >= rem keys)
      // the group's 32 bins over the cluster, lane 0 the top bin
      const int bin = gsel * 32 + 31 - lane;
      uint32_t part[kIxSelCtas];
#pragma unroll
      for (int r = 0; r < kIxSelCtas; ++r) part[r] = ix_peer(&cnt[pb][0], r)[bin];
      int cb = 0;
#pragma unroll
      for (int r = 0; r < kIxSelCtas; ++r) cb += (int)part[r];
      int binc = cb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v2 = __shfl_up_sync(0xffffffffu, binc, o);
        if (lane >= o) binc += v2;
      }
      const int babove = binc - cb;
      const unsigned hit = __ballot_sync(0xffffffffu, babove < grem && grem <= babove + cb);
      const int hl = hit ? __ffs(hit) - 1 : 0;
      const int b = __shfl_sync(0xffffffffu, bin, hl);
      const int brem = __shfl_sync(0xffffffffu, grem - babove, hl);
      // the chosen bin's smallest and largest image over the cluster
      mn = __reduce_min_sync(0xffffffffu, lane < kIxSelCtas ? *ix_peer(&bmin[pb][b], lane) : 0xFFFFFFFFu);
      mx = __reduce_max_sync(0xffffffffu, lane < kIxSelCtas ? *ix_peer(&bmax[pb][b], lane) : 0u);
      if (lane == 0) {
        s_lo = mn;
        s_hi = mx;
        s_rem = brem;
      }
    }
    __syncthreads();
    lo = s_lo;
    hi = s_hi;
    rem = s_rem;
  }
  if (lo < hi && rank == 0 && tid == 0) set_status(p.status, COLI_DEV_SELECT_ROUNDS);
  const uint32_t thr = lo;     // the topk-th largest image: topk - rem keys lie above it, `rem` equal keys are taken

  // per warp, a contiguous run of the CTA's keys: keys above the threshold and keys equal to it
  const int seg = ((n + nw - 1) / nw + 31) & ~31;
  const int w0 = min(n, wid * seg), w1 = min(n, w0 + seg);
  int n_above = 0, n_eq = 0;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint32_t u = i < w1 ? u_s[i] : 0u;
    n_above += __popc(__ballot_sync(0xffffffffu, i < w1 && u > thr));
    n_eq += __popc(__ballot_sync(0xffffffffu, i < w1 && u == thr));
  }
  // one scan of both counts, packed (each below 2^16: a CTA holds at most 16384 keys)
  const int packed_w = __shfl_sync(0xffffffffu, block_exclusive_scan(lane == 0 ? (n_eq << 16) | n_above : 0, warp_tot,
                                                                     &total), 0);
  const int eq_w = packed_w >> 16;
  const int eq_cta = total >> 16, above_cta = total & 0xFFFF;
  if (tid == 0) {
    ex[2] = (uint32_t)above_cta;
    ex[3] = (uint32_t)eq_cta;
  }
  ix_cluster_sync();                                      // (2) every CTA's counts are visible
  // keys the lower CTAs place (their keys above, and their share of the equal keys, lowest keys first):
  // lane r of warp 0 reads CTA r's counts, a warp scan orders them
  if (wid == 0) {
    const bool lower = lane < (int)rank;
    const int ab = lower ? (int)*ix_peer(&ex[2], lane) : 0, eq = lower ? (int)*ix_peer(&ex[3], lane) : 0;
    int inc = eq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t2 = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t2;
    }
    const int placed = ab + max(0, min(eq, rem - (inc - eq)));
    const int placed_sum = __reduce_add_sync(0xffffffffu, placed);
    const int eq_sum = __shfl_sync(0xffffffffu, inc, 31);
    if (lane == 0) {
      wmin[0] = (uint32_t)placed_sum;
      wmax[0] = (uint32_t)eq_sum;
    }
  }
  __syncthreads();
  const int placed_before = (int)wmin[0], eq_before = (int)wmax[0];
  const int eq_base = eq_before + eq_w;                   // equal keys below this warp's run
  const int take_w = max(0, min(n_eq, rem - eq_base));
  int pos = placed_before +
            __shfl_sync(0xffffffffu, block_exclusive_scan(lane == 0 ? n_above + take_w : 0, warp_tot, &total), 0);
  int eq_seen = eq_base;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint32_t u = i < w1 ? u_s[i] : 0u;
    const bool eq = i < w1 && u == thr;
    const unsigned em = __ballot_sync(0xffffffffu, eq);
    const bool take = i < w1 && (u > thr || (eq && eq_seen + __popc(em & ((1u << lane) - 1u)) < rem));
    const unsigned tm = __ballot_sync(0xffffffffu, take);
    if (take) {
      const int at = pos + __popc(tm & ((1u << lane) - 1u));
      if (at < topk) o[at] = k0 + i;                    // exactly topk keys are placed; the bound is a guard
    }
    pos += __popc(tm);
    eq_seen += __popc(em);
  }
  // (3) no CTA leaves while a peer may read it.  Relaxed: no data crosses this barrier, and every peer load
  // of this CTA's shared memory was consumed before its arrival; the index stores need no cluster release.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ host side

static cudaError_t launch_indexer_select(const IndexerCall& c, cudaStream_t st) {
  IxSel p;
  p.scores = c.scores;
  p.ls = c.L;
  p.L = c.L;
  p.pos0 = c.pos0;
  p.topk = c.topk;
  p.chunk = ((c.L + kIxSelCtas - 1) / kIxSelCtas + 31) & ~31;
  p.out = c.out;
  p.status = c.status;
  const size_t smem = (size_t)(6 * kIxBins + p.chunk) * 4;
  cudaError_t e = cudaFuncSetAttribute(indexer_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kIxSelCtas, c.T);
  cfg.blockDim = dim3(kIxSelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kIxSelCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, indexer_select_kernel, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_indexer(const IndexerCall& c, cudaStream_t st, int num_sms) {
  cudaError_t e = c.steps & 1 ? launch_indexer_scores(c, st, num_sms) : cudaSuccess;
  if (e == cudaSuccess && (c.steps & 2)) e = launch_indexer_select(c, st);
  return e;
}

cudaError_t launch_indexer_scores(const IndexerCall& c, cudaStream_t st, int num_sms) {
  auto encode = c.encode;
  const int n_groups = (c.T + kIxQMax - 1) / kIxQMax;
  const size_t smem = (size_t)kIxStages * kIxStageBytes + 2 * (kIxQMax * kIxHeads) * 128 + 1024;
  cudaError_t e = cudaFuncSetAttribute(indexer_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  CUtensorMap kmap;
  {
    const cuuint64_t gdim[2] = {(cuuint64_t)kIxD, (cuuint64_t)c.L};
    const cuuint64_t gstr[1] = {(cuuint64_t)kIxD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kIxKeys};
    const cuuint32_t es[2] = {1, 1};
    if (encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(c.keys), gdim, gstr, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int n_tiles = (c.L + kIxKeys - 1) / kIxKeys;
  const int grid = n_tiles < num_sms ? n_tiles : num_sms;
  for (int g = 0; g < n_groups; ++g) {
    const int t0 = g * kIxQMax, tq = c.T - t0 < kIxQMax ? c.T - t0 : kIxQMax;
    CUtensorMap qmap;
    const cuuint64_t gdim[2] = {(cuuint64_t)kIxD, (cuuint64_t)(tq * kIxHeads)};
    const cuuint64_t gstr[1] = {(cuuint64_t)kIxD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)(tq * kIxHeads)};
    const cuuint32_t es[2] = {1, 1};
    if (encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<uint16_t*>(static_cast<const uint16_t*>(c.q) + (size_t)t0 * kIxHeads * kIxD), gdim, gstr,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    IxArgs p;
    p.T = tq;
    p.L = c.L;
    p.pos0 = c.pos0 + t0;
    p.w = c.w + (size_t)t0 * kIxHeads;
    p.scores = c.scores + (size_t)t0 * c.L;
    p.ls = c.L;
    p.status = c.status;
    p.wait_ns = c.wait_ns;
    indexer_scores_kernel<<<grid, kIxThreads, smem, st>>>(p, kmap, qmap);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace coli
