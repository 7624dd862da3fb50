// Expert-slot cache in HBM with a host-memory tier.
//
// "25GB RAM runs 744B GLM-5.2" page (pwwt.cn), section 2: the engine spreads
// the weights over a hierarchy of storage tiers and reads the routed experts
// a layer needs on demand; section 3.5: a per-layer LRU cache of experts, with
// the next experts read ahead asynchronously.  "Colibri walkthrough" page
// (discosf.com), section 3.1: the cache unit is an "expert slot" holding one
// expert's whole weights; each slot keeps a last_used timestamp and a
// hit_count, and eviction prefers slots with a low hit_count and an old
// last_used (a frequency-weighted LRU); the engine reports cache_hit_rate.
//
// Here the lower tier is host memory (reached over the GPU's host link) and
// the upper tier is a pool of slots in device memory.  A cached forward runs
// the router on the GPU, reads the list of chosen experts back, admits them
// (hits keep their slot; misses are copied into a victim slot with one
// cudaMemcpyAsync per packed array), uploads the expert -> slot table and runs
// the expert kernels on the slots.  The expert kernels are those of the
// resident path, so the outputs are the same, bit for bit.
//
// Eviction (the reading of "low hit_count and old last_used"): among the slots
// the current forward does not use, an empty slot first, else the one with
// the smallest last_used + weight * hit_count, where hit_count counts the
// forwards that used the expert since it entered the slot: every use buys
// `weight` steps of recency.  weight = 0 is plain LRU.  Ties go to the smaller
// last_used, then the lower slot index.
#include <cstring>
#include <vector>

#include "plan.h"

using namespace coli;

namespace {

// The slot policy, host only (shared by the cache and the simulator).
struct SlotPolicy {
  int E = 0, n_slots = 0;
  double weight = 0.0;
  long long step = 0;
  std::vector<int> slot_expert;        // expert id or -1
  std::vector<long long> last_used;
  std::vector<long long> hit_count;
  std::vector<int> expert_slot;        // slot or -1
  std::vector<char> busy;              // used by the forward being admitted

  void init(int e, int s, double w) {
    E = e;
    n_slots = s;
    weight = w;
    step = 0;
    slot_expert.assign(s, -1);
    last_used.assign(s, 0);
    hit_count.assign(s, 0);
    expert_slot.assign(e, -1);
    busy.assign(s, 0);
  }

  int victim() const {
    int best = -1;
    double bp = 0.0;
    for (int i = 0; i < n_slots; ++i) {
      if (busy[i]) continue;
      if (slot_expert[i] < 0) return i;
      const double p = (double)last_used[i] + weight * (double)hit_count[i];
      if (best < 0 || p < bp || (p == bp && last_used[i] < last_used[best])) {
        best = i;
        bp = p;
      }
    }
    return best;
  }

  // Admit the experts of one forward (distinct ids).  on_miss(expert, slot, evicted expert or -1) is
  // called for each expert that has to be loaded.  Returns the hits, or -1 if they cannot all be held.
  template <class OnMiss>
  int admit(const int* ids, int n, OnMiss on_miss) {
    if (n > n_slots) return -1;
    ++step;
    std::fill(busy.begin(), busy.end(), 0);
    int hits = 0;
    for (int i = 0; i < n; ++i) {
      const int s = expert_slot[ids[i]];
      if (s >= 0) {
        busy[s] = 1;
        last_used[s] = step;
        ++hit_count[s];
        ++hits;
      }
    }
    for (int i = 0; i < n; ++i) {
      const int e = ids[i];
      if (expert_slot[e] >= 0) continue;
      const int s = victim();
      const int old = slot_expert[s];
      if (old >= 0) expert_slot[old] = -1;
      slot_expert[s] = e;
      expert_slot[e] = s;
      last_used[s] = step;
      hit_count[s] = 1;
      busy[s] = 1;
      on_miss(e, s, old);
    }
    return hits;
  }

  // Bring experts in ahead of their use (no recency or count of their own yet): prefetch_begin, then
  // prefetch per expert, which returns its slot and whether it had to be loaded (-1: every slot is taken
  // by this batch).  The experts of one batch do not evict each other.
  void prefetch_begin() { std::fill(busy.begin(), busy.end(), 0); }
  int prefetch(int e, bool& loaded, int& evicted) {
    loaded = false;
    evicted = -1;
    if (expert_slot[e] >= 0) {
      busy[expert_slot[e]] = 1;
      return expert_slot[e];
    }
    const int s = victim();
    if (s < 0) return -1;
    evicted = slot_expert[s];
    if (evicted >= 0) expert_slot[evicted] = -1;
    slot_expert[s] = e;
    expert_slot[e] = s;
    last_used[s] = step;
    hit_count[s] = 0;
    busy[s] = 1;
    loaded = true;
    return s;
  }
};

}  // namespace

struct coli_cache {
  coli_moe_plan* plan = nullptr;
  SlotPolicy pol;
  size_t slot_bytes = 0;
  size_t off[9] = {0}, len[9] = {0};   // gate q/s/z, up q/s/z, down q/s/z within a slot
  uint8_t* slots = nullptr;            // caller's device memory
  std::vector<coli_expert> host;       // [E] host-memory arrays of every routed expert
  DevExpert* d_experts = nullptr;      // [n_slots + 1] (the last one: the resident shared expert)
  CUtensorMap* d_maps = nullptr;       // [(n_slots + 1) * 6]
  int32_t* d_slot_of = nullptr;        // [E + 1]
  int32_t* h_slot_of = nullptr;        // pinned [E + 1]
  int32_t* h_unique = nullptr;         // pinned [E + 2]
  coli_cache_stats stats;
  coli_status err = COLI_OK;
  int pilot_n = 0;                     // experts of the last pilot prediction
};

static void slot_layout(const coli_moe_desc& d, size_t* off, size_t* len, size_t* total) {
  size_t o = 0;
  for (int m = 0; m < 3; ++m) {
    const size_t N = m < 2 ? d.d_ff : d.d, K = m < 2 ? d.d : d.d_ff;
    size_t q, s, z;
    if (d.qtype == COLI_Q_INT4_G128) {
      q = N * K / 2;
      s = N * (K / 128) * 2;
      z = N * ((K / 128 + 1) / 2);
    } else {
      q = N * K;
      s = N * 4;
      z = N;
    }
    const size_t parts[3] = {q, s, z};
    for (int j = 0; j < 3; ++j) {
      off[3 * m + j] = o;
      len[3 * m + j] = parts[j];
      o = align_up(o + parts[j], 256);
    }
  }
  *total = o;
}

static coli_status copy_expert(coli_cache* c, int e, int slot, cudaStream_t st) {
  const coli_expert& h = c->host[e];
  const coli_qmat* mats[3] = {&h.gate, &h.up, &h.down};
  uint8_t* base = c->slots + (size_t)slot * c->slot_bytes;
  // an expert stored in host memory in the slot's own layout moves in one copy
  const uint8_t* h0 = static_cast<const uint8_t*>(h.gate.q);
  bool packed = true;
  for (int m = 0; m < 3; ++m) {
    const void* src[3] = {mats[m]->q, mats[m]->scale, mats[m]->zp};
    for (int j = 0; j < 3; ++j) packed &= static_cast<const uint8_t*>(src[j]) == h0 + c->off[3 * m + j];
  }
  if (packed) {
    const cudaError_t ce = cudaMemcpyAsync(base, h0, c->slot_bytes, cudaMemcpyHostToDevice, st);
    if (ce != cudaSuccess) return cuda_fail(ce, "expert cache: copy from host memory");
    c->stats.bytes_copied += (long long)c->slot_bytes;
    return COLI_OK;
  }
  for (int m = 0; m < 3; ++m) {
    const void* src[3] = {mats[m]->q, mats[m]->scale, mats[m]->zp};
    for (int j = 0; j < 3; ++j) {
      const cudaError_t ce =
          cudaMemcpyAsync(base + c->off[3 * m + j], src[j], c->len[3 * m + j], cudaMemcpyHostToDevice, st);
      if (ce != cudaSuccess) return cuda_fail(ce, "expert cache: copy from host memory");
    }
  }
  c->stats.bytes_copied += (long long)c->slot_bytes;
  return COLI_OK;
}

// Between routing and the expert kernels: read the chosen experts back, admit them, upload the table.
static coli_status cache_between(void* ctx, const FwdArgs& a, cudaStream_t st) {
  coli_cache* c = static_cast<coli_cache*>(ctx);
  const int E = a.E;
  cudaError_t ce = cudaMemcpyAsync(c->h_unique, a.n_unique, 4, cudaMemcpyDeviceToHost, st);
  if (ce == cudaSuccess) ce = cudaMemcpyAsync(c->h_unique + 1, a.unique, (size_t)E * 4, cudaMemcpyDeviceToHost, st);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(st);
  if (ce != cudaSuccess) return cuda_fail(ce, "expert cache: read the chosen experts");
  const int nu = c->h_unique[0];
  if (nu < 0 || nu > E) return fail(COLI_EDEVICE, "expert cache: routing reported %d experts", nu);
  for (int i = 0; i < nu; ++i)
    if (c->h_unique[1 + i] < 0 || c->h_unique[1 + i] >= E) return fail(COLI_EDEVICE, "expert cache: bad expert id");
  c->err = COLI_OK;
  const int hits = c->pol.admit(c->h_unique + 1, nu, [&](int e, int s, int evicted) {
    if (evicted >= 0) ++c->stats.evictions;
    if (c->err == COLI_OK) c->err = copy_expert(c, e, s, st);
  });
  if (hits < 0)
    return fail(COLI_EUNSUPPORTED, "expert cache: this forward needs %d experts, the cache has %d slots", nu,
                c->pol.n_slots);
  if (c->err != COLI_OK) return c->err;
  c->stats.forwards += 1;
  c->stats.lookups += nu;
  c->stats.hits += hits;
  c->stats.misses += nu - hits;
  for (int i = 0; i < nu; ++i) c->h_slot_of[c->h_unique[1 + i]] = c->pol.expert_slot[c->h_unique[1 + i]];
  c->h_slot_of[E] = c->pol.n_slots;
  ce = cudaMemcpyAsync(c->d_slot_of, c->h_slot_of, ((size_t)E + 1) * 4, cudaMemcpyHostToDevice, st);
  return ce == cudaSuccess ? COLI_OK : cuda_fail(ce, "expert cache: upload the slot table");
}

extern "C" {

coli_status colibri_moe_cache_slot_bytes(const coli_moe_plan_t* plan, size_t* bytes) {
  if (!plan || !bytes) return fail(COLI_EINVAL, "cache_slot_bytes: null argument");
  size_t off[9], len[9];
  slot_layout(plan->desc, off, len, bytes);
  return COLI_OK;
}

coli_status colibri_moe_cache_create(coli_moe_plan_t* plan, int n_slots, double weight, const coli_expert* host_experts,
                                     const coli_expert* shared, void* slot_memory, size_t slot_memory_bytes,
                                     coli_cache_t** cache) {
  if (!plan || !host_experts || !slot_memory || !cache) return fail(COLI_EINVAL, "cache_create: null argument");
  const coli_moe_desc& d = plan->desc;
  if (n_slots < 1) return fail(COLI_EINVAL, "cache_create: n_slots must be positive");
  if (!(weight >= 0.0)) return fail(COLI_EINVAL, "cache_create: weight must be >= 0");
  if (d.has_shared && !shared) return fail(COLI_EINVAL, "cache_create: plan has a shared expert but shared is NULL");
  if (!d.has_shared && shared) return fail(COLI_EINVAL, "cache_create: plan has no shared expert");
  if (!aligned(slot_memory, 256)) return fail(COLI_EALIGN, "cache_create: slot memory not 256-byte aligned");
  coli_cache* c = new (std::nothrow) coli_cache();
  if (!c) return fail(COLI_EINVAL, "cache_create: out of host memory");
  slot_layout(d, c->off, c->len, &c->slot_bytes);
  if (slot_memory_bytes < (size_t)n_slots * c->slot_bytes) {
    const size_t need = (size_t)n_slots * c->slot_bytes;
    delete c;
    return fail(COLI_EWORKSPACE, "cache_create: slot memory %zu bytes < %zu needed", slot_memory_bytes, need);
  }
  for (int e = 0; e < d.E; ++e) {
    const coli_expert& h = host_experts[e];
    const coli_qmat* mats[3] = {&h.gate, &h.up, &h.down};
    for (int m = 0; m < 3; ++m)
      if (!mats[m]->q || !mats[m]->scale || !mats[m]->zp) {
        delete c;
        return fail(COLI_EINVAL, "cache_create: host expert %d matrix %d has a null pointer", e, m);
      }
  }
  c->plan = plan;
  c->slots = static_cast<uint8_t*>(slot_memory);
  c->host.assign(host_experts, host_experts + d.E);
  c->pol.init(d.E, n_slots, weight);
  memset(&c->stats, 0, sizeof(c->stats));
  // descriptors and maps of every slot (fixed device addresses) and of the resident shared expert
  std::vector<DevExpert> hx((size_t)n_slots + 1);
  std::vector<CUtensorMap> hm(((size_t)n_slots + 1) * 6);
  memset(hx.data(), 0, hx.size() * sizeof(DevExpert));
  memset(hm.data(), 0, hm.size() * sizeof(CUtensorMap));
  coli_status rc = COLI_OK;
  for (int s = 0; s <= n_slots && rc == COLI_OK; ++s) {
    coli_expert ex;
    int F = d.d_ff;
    if (s < n_slots) {
      uint8_t* b = c->slots + (size_t)s * c->slot_bytes;
      coli_qmat* mats[3] = {&ex.gate, &ex.up, &ex.down};
      for (int m = 0; m < 3; ++m) {
        mats[m]->q = b + c->off[3 * m];
        mats[m]->scale = b + c->off[3 * m + 1];
        mats[m]->zp = b + c->off[3 * m + 2];
      }
    } else if (d.has_shared) {
      ex = *shared;
      F = d.shared_d_ff;
    } else {
      break;
    }
    rc = encode_expert(d, F, ex, s, hx[s], &hm[(size_t)s * 3], &hm[((size_t)n_slots + 1) * 3 + (size_t)s * 3]);
  }
  cudaError_t ce = cudaSuccess;
  if (rc == COLI_OK) {
    ce = cudaMalloc(&c->d_experts, hx.size() * sizeof(DevExpert));
    if (ce == cudaSuccess) ce = cudaMalloc(&c->d_maps, hm.size() * sizeof(CUtensorMap));
    if (ce == cudaSuccess) ce = cudaMalloc(&c->d_slot_of, ((size_t)d.E + 1) * 4);
    if (ce == cudaSuccess) ce = cudaHostAlloc(&c->h_slot_of, ((size_t)d.E + 1) * 4, cudaHostAllocDefault);
    if (ce == cudaSuccess) ce = cudaHostAlloc(&c->h_unique, ((size_t)d.E + 2) * 4, cudaHostAllocDefault);
    if (ce == cudaSuccess)
      ce = cudaMemcpy(c->d_experts, hx.data(), hx.size() * sizeof(DevExpert), cudaMemcpyHostToDevice);
    if (ce == cudaSuccess) ce = cudaMemcpy(c->d_maps, hm.data(), hm.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice);
    if (ce != cudaSuccess) rc = cuda_fail(ce, "cache_create: device tables");
  }
  if (rc != COLI_OK) {
    colibri_moe_cache_destroy(c);
    return rc;
  }
  for (int e = 0; e <= d.E; ++e) c->h_slot_of[e] = e == d.E ? n_slots : 0;
  *cache = c;
  return COLI_OK;
}

coli_status colibri_moe_forward_cached(coli_moe_plan_t* plan, coli_cache_t* cache, int T, const void* x,
                                       const float* router_w, const float* bias, const float* residual, float* out,
                                       void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan || !cache) return fail(COLI_EINVAL, "forward_cached: null argument");
  if (cache->plan != plan) return fail(COLI_EINVAL, "forward_cached: the cache belongs to another plan");
  const ExpertTables tb{cache->d_experts, cache->d_maps, cache->pol.n_slots, cache->d_slot_of};
  return forward_impl(plan, tb, cache_between, cache, T, x, router_w, bias, residual, out, workspace,
                      workspace_bytes, stream);
}

coli_status colibri_moe_cache_prefetch(coli_cache_t* cache, const int32_t* experts, int n, void* stream) {
  if (!cache || (n > 0 && !experts)) return fail(COLI_EINVAL, "cache_prefetch: null argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cache->pol.prefetch_begin();
  for (int i = 0; i < n; ++i) {
    const int e = experts[i];
    if (e < 0 || e >= cache->pol.E) return fail(COLI_EINVAL, "cache_prefetch: expert id %d out of range", e);
    bool loaded = false;
    int evicted = -1;
    const int s = cache->pol.prefetch(e, loaded, evicted);
    if (s < 0) return fail(COLI_EUNSUPPORTED, "cache_prefetch: no free slot");
    if (!loaded) continue;
    if (evicted >= 0) ++cache->stats.evictions;
    ++cache->stats.prefetched;
    const coli_status rc = copy_expert(cache, e, s, st);
    if (rc != COLI_OK) return rc;
  }
  return COLI_OK;
}

// Routing-only pass of the next layer: read its chosen experts back and prefetch them.
static coli_status pilot_between(void* ctx, const FwdArgs& a, cudaStream_t st) {
  coli_cache* c = static_cast<coli_cache*>(ctx);
  const int E = a.E;
  cudaError_t ce = cudaMemcpyAsync(c->h_unique, a.n_unique, 4, cudaMemcpyDeviceToHost, st);
  if (ce == cudaSuccess) ce = cudaMemcpyAsync(c->h_unique + 1, a.unique, (size_t)E * 4, cudaMemcpyDeviceToHost, st);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(st);
  if (ce != cudaSuccess) return cuda_fail(ce, "cache_pilot: read the predicted experts");
  const int nu = c->h_unique[0];
  if (nu < 0 || nu > E) return fail(COLI_EDEVICE, "cache_pilot: routing reported %d experts", nu);
  c->pilot_n = nu;
  const int take = nu < c->pol.n_slots ? nu : c->pol.n_slots;
  c->stats.predicted += nu;
  const coli_status rc = colibri_moe_cache_prefetch(c, c->h_unique + 1, take, st);
  return rc == COLI_OK ? kStopAfterRouting : rc;
}

coli_status colibri_moe_cache_pilot(coli_moe_plan_t* plan_next, coli_cache_t* cache_next, int T, const void* x,
                                    const float* router_w, const float* bias, int32_t* predicted, int* n_predicted,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan_next || !cache_next) return fail(COLI_EINVAL, "cache_pilot: null argument");
  if (cache_next->plan != plan_next) return fail(COLI_EINVAL, "cache_pilot: the cache belongs to another plan");
  const ExpertTables tb{cache_next->d_experts, cache_next->d_maps, cache_next->pol.n_slots, cache_next->d_slot_of};
  const coli_status rc = forward_impl(plan_next, tb, pilot_between, cache_next, T, x, router_w, bias, nullptr,
                                      reinterpret_cast<float*>(workspace), workspace, workspace_bytes, stream);
  if (rc != COLI_OK) return rc;
  if (n_predicted) *n_predicted = cache_next->pilot_n;
  if (predicted)
    for (int i = 0; i < cache_next->pilot_n; ++i) predicted[i] = cache_next->h_unique[1 + i];
  return COLI_OK;
}

coli_status colibri_moe_cache_stats(const coli_cache_t* cache, coli_cache_stats* stats) {
  if (!cache || !stats) return fail(COLI_EINVAL, "cache_stats: null argument");
  *stats = cache->stats;
  return COLI_OK;
}

coli_status colibri_moe_cache_reset_stats(coli_cache_t* cache) {
  if (!cache) return fail(COLI_EINVAL, "cache_reset_stats: null argument");
  memset(&cache->stats, 0, sizeof(cache->stats));
  return COLI_OK;
}

coli_status colibri_moe_cache_resident(const coli_cache_t* cache, int32_t* slot_of_expert) {
  if (!cache || !slot_of_expert) return fail(COLI_EINVAL, "cache_resident: null argument");
  for (int e = 0; e < cache->pol.E; ++e) slot_of_expert[e] = cache->pol.expert_slot[e];
  return COLI_OK;
}

void colibri_moe_cache_destroy(coli_cache_t* cache) {
  if (!cache) return;
  cudaFree(cache->d_experts);
  cudaFree(cache->d_maps);
  cudaFree(cache->d_slot_of);
  cudaFreeHost(cache->h_slot_of);
  cudaFreeHost(cache->h_unique);
  delete cache;
}

coli_status colibri_moe_cache_simulate(int E, int n_slots, double weight, const int32_t* expert_sets,
                                       const int32_t* set_sizes, int n_steps, int64_t* hits, int64_t* misses) {
  if (E < 1 || n_slots < 1 || n_steps < 0 || !(weight >= 0.0) || (n_steps > 0 && (!expert_sets || !set_sizes)) ||
      !hits || !misses)
    return fail(COLI_EINVAL, "cache_simulate: bad argument");
  SlotPolicy pol;
  pol.init(E, n_slots, weight);
  *hits = *misses = 0;
  const int32_t* p = expert_sets;
  for (int t = 0; t < n_steps; ++t) {
    const int n = set_sizes[t];
    for (int i = 0; i < n; ++i)
      if (p[i] < 0 || p[i] >= E) return fail(COLI_EINVAL, "cache_simulate: expert id out of range");
    const int h = pol.admit(p, n, [](int, int, int) {});
    if (h < 0) return fail(COLI_EUNSUPPORTED, "cache_simulate: step %d needs %d experts, %d slots", t, n, n_slots);
    *hits += h;
    *misses += n - h;
    p += n;
  }
  return COLI_OK;
}

}  // extern "C"
