// C ABI of the quantized sparse MoE layer library: plan validation, expert
// binding (TMA tensor maps + device descriptor table), the forward launch
// sequence, routing debug copies, status read-back and per-kernel timing.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "plan.h"

using namespace coli;

namespace {
thread_local std::string g_err;
}  // namespace

namespace coli {

coli_status fail(coli_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

coli_status cuda_fail(cudaError_t e, const char* what) {
  return fail(COLI_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

}  // namespace coli

namespace {

enum KernelId {
  K_ROUTE = 0, K_ROUTER, K_TOPK, K_PERMUTE, K_PREP, K_GATEUP, K_DOWN, K_GATHER, K_TILES, K_TC_GATEUP, K_TC_DOWN,
  K_COMBINE, K_RSPLIT, K_COUNT
};
const char* kKernelNames[K_COUNT] = {"route_decode", "router_logits",  "router_topk",    "permute",
                                     "quantize_h",   "expert_gate_up", "expert_down",    "gather_x",
                                     "plan_tiles",   "tc_gate_up",     "tc_down",        "combine",
                                     "router_split"};

}  // namespace

namespace coli {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

static int matrix_row_bytes(int qtype, int K) { return qtype == COLI_Q_INT4_G128 ? K / 2 : K; }

coli_status encode_expert(const coli_moe_desc& d, int F, const coli_expert& ex, int id, DevExpert& dx,
                          CUtensorMap* dec, CUtensorMap* tc) {
  auto encode = get_encode();
  if (!encode) return fail(COLI_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const size_t sal = d.qtype == COLI_Q_INT4_G128 ? 2 : 4;
  const coli_qmat* mats[3] = {&ex.gate, &ex.up, &ex.down};
  for (int m = 0; m < 3; ++m) {
    const coli_qmat& qm = *mats[m];
    if (!qm.q || !qm.scale || !qm.zp) return fail(COLI_EINVAL, "expert %d matrix %d has a null pointer", id, m);
    if (!aligned(qm.q, 16)) return fail(COLI_EALIGN, "expert %d matrix %d codes not 16-byte aligned", id, m);
    if (!aligned(qm.scale, sal)) return fail(COLI_EALIGN, "expert %d matrix %d scales misaligned", id, m);
    const int N = m < 2 ? F : d.d, K = m < 2 ? d.d : F;
    DevMat& dm = dx.m[m];
    dm.q = static_cast<const uint8_t*>(qm.q);
    dm.s = qm.scale;
    dm.z = static_cast<const uint8_t*>(qm.zp);
    dm.N = N;
    dm.K = K;
    const cuuint64_t row_bytes = (cuuint64_t)matrix_row_bytes(d.qtype, K);
    const cuuint64_t gdim[2] = {row_bytes, (cuuint64_t)N};
    const cuuint64_t gstride[1] = {row_bytes};
    // box width: 256 bytes, or the whole row when rows are shorter (128 bytes)
    const cuuint32_t boxw = row_bytes < (cuuint64_t)kTmaBoxBytes ? (cuuint32_t)row_bytes : (cuuint32_t)kTmaBoxBytes;
    const cuuint32_t box[2] = {boxw, (cuuint32_t)(m < 2 ? kGateUpBoxRows : kDownBoxRows)};
    const cuuint32_t estride[2] = {1, 1};
    CUresult r = encode(&dec[m], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(qm.q), gdim, gstride, box,
                        estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(COLI_ECUDA, "cuTensorMapEncodeTiled failed (%d) for expert %d", (int)r, id);
    // tensor-core path: one pipeline stage of codes (32, 64 or 128 bytes) x 128 rows, stored with
    // the swizzle of the same width so that the dequantising threads read rows without bank conflicts
    const int pf_row = prefill_raw_row_bytes(d.qtype, m < 2);
    const cuuint32_t box2[2] = {(cuuint32_t)pf_row, (cuuint32_t)kPrefillRows};
    const CUtensorMapSwizzle swz = pf_row == 32   ? CU_TENSOR_MAP_SWIZZLE_32B
                                   : pf_row == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                  : CU_TENSOR_MAP_SWIZZLE_128B;
    r = encode(&tc[m], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(qm.q), gdim, gstride, box2, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(COLI_ECUDA, "cuTensorMapEncodeTiled (tensor-core box) failed (%d)", (int)r);
  }
  dx.F = F;
  return COLI_OK;
}

}  // namespace coli

extern "C" {

const char* colibri_moe_last_error(void) { return g_err.c_str(); }

coli_status colibri_moe_plan(const coli_moe_desc* desc, coli_moe_plan_t** plan, size_t* workspace_bytes) {
  if (!desc || !plan || !workspace_bytes) return fail(COLI_EINVAL, "plan: null argument");
  const coli_moe_desc& d = *desc;
  if (d.T_max < 1 || d.d < 1 || d.d_ff < 1 || d.E < 1 || d.k < 1)
    return fail(COLI_EINVAL, "plan: T_max, d, d_ff, E, k must be positive");
  if (d.E > kMaxE) return fail(COLI_EUNSUPPORTED, "plan: E=%d exceeds %d", d.E, kMaxE);
  if (d.k > d.E || d.k > kMaxK) return fail(COLI_EINVAL, "plan: need 1 <= k <= min(E, %d)", kMaxK);
  if (d.qtype != COLI_Q_INT4_G128 && d.qtype != COLI_Q_INT8_PC) return fail(COLI_EUNSUPPORTED, "plan: unknown qtype");
  if (d.xtype != COLI_X_BF16 && d.xtype != COLI_X_F32) return fail(COLI_EUNSUPPORTED, "plan: unknown xtype");
  if (d.has_shared != 0 && d.has_shared != 1) return fail(COLI_EINVAL, "plan: has_shared must be 0 or 1");
  if (d.has_shared && d.shared_d_ff < 1) return fail(COLI_EINVAL, "plan: shared_d_ff must be positive");
  const int mult = d.qtype == COLI_Q_INT4_G128 ? 256 : 128;
  if (d.d % mult || d.d_ff % mult || (d.has_shared && d.shared_d_ff % mult))
    return fail(COLI_EUNSUPPORTED, "plan: d and FFN sizes must be multiples of %d for this qtype", mult);
  if ((long long)d.T_max * d.k > (1LL << 30)) return fail(COLI_EUNSUPPORTED, "plan: T_max*k too large");
  if (!(d.routed_scale == d.routed_scale)) return fail(COLI_EINVAL, "plan: routed_scale is NaN");

  coli_moe_plan* p = new (std::nothrow) coli_moe_plan();
  if (!p) return fail(COLI_EINVAL, "plan: out of host memory");
  p->desc = d;
  p->Fmax = d.has_shared && d.shared_d_ff > d.d_ff ? d.shared_d_ff : d.d_ff;
  const size_t T = (size_t)d.T_max, k = (size_t)d.k, E = (size_t)d.E;
  const size_t P = T * k, rows = P + (d.has_shared ? T : 0);
  WsLayout& w = p->ws;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  w.status = take(64);
  w.topk_idx = take(T * k * 4);
  w.topk_w = take(T * k * 4);
  w.near_tie = take(T * 4);
  w.offsets = take((E + 2) * 4);
  w.pair_token = take(rows * 4);
  w.pair_slot = take(P * 4);
  w.pair_of = take(P * 4);
  w.unique = take((E + 1) * 4);
  w.utab = take((E + 1) * 16);
  w.n_unique = take(16);
  w.logits = take((size_t)kRouterKSplit * T * E * 4);
  w.xs = take(T * (size_t)d.d * 4);
  w.xsum = take(T * (size_t)(d.d / kXsumBlock) * 4);
  w.xq = take(T * (size_t)d.d * 2);
  w.xqs = take(T * (size_t)(d.d / kXqBlock) * 8);
  w.h = take(rows * (size_t)p->Fmax * 4);
  w.hsum = take(rows * (size_t)(p->Fmax / 8) * 4);
  w.hq = take(rows * (size_t)p->Fmax * 2);
  w.hqs = take(rows * (size_t)(p->Fmax / kXqBlock) * 8);
  w.y = take(rows * (size_t)d.d * 4);
  w.xh = w.chunks = w.gu_tiles = w.dn_tiles = w.pf_counts = w.wsplit = 0;
  if (d.T_max > kDecodeMaxT) {
    const size_t max_chunks = (E + 1) + rows / kPrefillChunk + 2;
    w.xh = take(rows * (size_t)d.d * 2);
    w.chunks = take(max_chunks * 16);
    w.gu_tiles = take(max_chunks * (size_t)(p->Fmax / kPrefillRows) * 16);
    w.dn_tiles = take(max_chunks * (size_t)(d.d / kPrefillRows) * 16);
    w.pf_counts = take(16);
    if (d.xtype == COLI_X_BF16 && d.T_max >= kRouterTcMinT && (d.d / kRouterKSplit) % 64 == 0)
      w.wsplit = take(3 * E * (size_t)d.d * 2);
  }
  w.total = off;
  *workspace_bytes = off;
  *plan = p;
  return COLI_OK;
}

void colibri_moe_destroy(coli_moe_plan_t* plan) {
  if (!plan) return;
  if (plan->device >= 0) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != plan->device) cudaSetDevice(plan->device);
    cudaFree(plan->d_experts);
    cudaFree(plan->d_maps);
    for (cudaEvent_t e : plan->prof_events) cudaEventDestroy(e);
    if (cur >= 0 && cur != plan->device) cudaSetDevice(cur);
  }
  delete plan;
}

coli_status colibri_moe_bind_experts(coli_moe_plan_t* plan, const coli_expert* experts, const coli_expert* shared) {
  if (!plan || !experts) return fail(COLI_EINVAL, "bind: null argument");
  const coli_moe_desc& d = plan->desc;
  if (d.has_shared && !shared) return fail(COLI_EINVAL, "bind: plan has a shared expert but shared is NULL");
  if (!d.has_shared && shared) return fail(COLI_EINVAL, "bind: plan has no shared expert");
  auto encode = get_encode();
  if (!encode) return fail(COLI_ECUDA, "bind: cuTensorMapEncodeTiled is not available from the driver");
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce, "bind: cudaGetDevice");
  int sms = 0;
  ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (ce != cudaSuccess) return cuda_fail(ce, "bind: cudaDeviceGetAttribute");

  const int slots = d.E + (d.has_shared ? 1 : 0);
  std::vector<DevExpert> hx((size_t)d.E + 1);
  std::vector<CUtensorMap> hm(((size_t)d.E + 1) * 6);   // [0, 3(E+1)): dequant-GEMV boxes; then tensor-core boxes
  memset(hx.data(), 0, hx.size() * sizeof(DevExpert));
  memset(hm.data(), 0, hm.size() * sizeof(CUtensorMap));
  for (int s = 0; s < slots; ++s) {
    const coli_expert& ex = s < d.E ? experts[s] : *shared;
    const coli_status rc = encode_expert(d, s < d.E ? d.d_ff : d.shared_d_ff, ex, s, hx[s], &hm[(size_t)s * 3],
                                         &hm[((size_t)d.E + 1) * 3 + (size_t)s * 3]);
    if (rc != COLI_OK) return rc;
  }
  if (plan->device >= 0 && plan->device != dev)
    return fail(COLI_ESTATE, "bind: plan was bound on device %d, current device is %d", plan->device, dev);
  if (!plan->d_experts) {
    ce = cudaMalloc(&plan->d_experts, hx.size() * sizeof(DevExpert));
    if (ce != cudaSuccess) return cuda_fail(ce, "bind: cudaMalloc(descriptors)");
    ce = cudaMalloc(&plan->d_maps, hm.size() * sizeof(CUtensorMap));
    if (ce != cudaSuccess) return cuda_fail(ce, "bind: cudaMalloc(tensor maps)");
  }
  ce = cudaMemcpy(plan->d_experts, hx.data(), hx.size() * sizeof(DevExpert), cudaMemcpyHostToDevice);
  if (ce != cudaSuccess) return cuda_fail(ce, "bind: upload descriptors");
  ce = cudaMemcpy(plan->d_maps, hm.data(), hm.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice);
  if (ce != cudaSuccess) return cuda_fail(ce, "bind: upload tensor maps");
  plan->device = dev;
  plan->num_sms = sms;
  plan->bound = true;
  return COLI_OK;
}

coli_status colibri_moe_forward(const coli_moe_plan_t* plan_c, int T, const void* x, const float* router_w,
                                const float* bias, const float* residual, float* out, void* workspace,
                                size_t workspace_bytes, void* stream) {
  coli_moe_plan_t* plan = const_cast<coli_moe_plan_t*>(plan_c);
  if (!plan) return fail(COLI_EINVAL, "forward: null plan");
  const ExpertTables tb{plan->d_experts, plan->d_maps, plan->desc.E, nullptr};
  return forward_impl(plan, tb, nullptr, nullptr, T, x, router_w, bias, residual, out, workspace, workspace_bytes,
                      stream);
}

}  // extern "C"

coli_status coli::forward_impl(coli_moe_plan* plan, const ExpertTables& tb, BetweenFn between, void* ctx, int T,
                               const void* x, const float* router_w, const float* bias, const float* residual,
                               float* out, void* workspace, size_t workspace_bytes, void* stream) {
  const coli_moe_desc& d = plan->desc;
  if (!plan->bound) return fail(COLI_ESTATE, "forward: experts not bound (call colibri_moe_bind_experts)");
  if (T < 1 || T > d.T_max) return fail(COLI_EINVAL, "forward: T=%d outside [1, %d]", T, d.T_max);
  if (!x || !router_w || !bias || !out || !workspace) return fail(COLI_EINVAL, "forward: null pointer");
  if (workspace_bytes < plan->ws.total)
    return fail(COLI_EWORKSPACE, "forward: workspace %zu bytes < required %zu", workspace_bytes, plan->ws.total);
  if (!aligned(workspace, 256)) return fail(COLI_EALIGN, "forward: workspace not 256-byte aligned");
  if (!aligned(x, 16) || !aligned(router_w, 16) || !aligned(out, 16) || (residual && !aligned(residual, 16)))
    return fail(COLI_EALIGN, "forward: x, router_w, residual and out must be 16-byte aligned");
  if (!aligned(bias, 4)) return fail(COLI_EALIGN, "forward: bias misaligned");

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const WsLayout& w = plan->ws;
  FwdArgs a;
  memset(&a, 0, sizeof(a));
  a.experts = tb.experts;
  a.maps = tb.maps;
  a.slot_of = tb.slot_of;
  a.T = T;
  a.d = d.d;
  a.F = d.d_ff;
  a.Fs = d.has_shared ? d.shared_d_ff : 0;
  a.E = d.E;
  a.k = d.k;
  a.qtype = d.qtype;
  a.xtype = d.xtype;
  a.has_shared = d.has_shared;
  a.rho = d.routed_scale;
  a.Fmax = plan->Fmax;
  a.x = x;
  a.router_w = router_w;
  a.bias = bias;
  a.residual = residual;
  a.out = out;
  a.status = reinterpret_cast<int32_t*>(ws + w.status);
  a.topk_idx = reinterpret_cast<int32_t*>(ws + w.topk_idx);
  a.topk_w = reinterpret_cast<float*>(ws + w.topk_w);
  a.near_tie = reinterpret_cast<int32_t*>(ws + w.near_tie);
  a.offsets = reinterpret_cast<int32_t*>(ws + w.offsets);
  a.pair_token = reinterpret_cast<int32_t*>(ws + w.pair_token);
  a.pair_slot = reinterpret_cast<int32_t*>(ws + w.pair_slot);
  a.pair_of = reinterpret_cast<int32_t*>(ws + w.pair_of);
  a.unique = reinterpret_cast<int32_t*>(ws + w.unique);
  a.utab = reinterpret_cast<int4*>(ws + w.utab);
  a.n_unique = reinterpret_cast<int32_t*>(ws + w.n_unique);
  a.logits = reinterpret_cast<float*>(ws + w.logits);
  a.xs = reinterpret_cast<float*>(ws + w.xs);
  a.xsum = reinterpret_cast<float*>(ws + w.xsum);
  a.xq = reinterpret_cast<uint32_t*>(ws + w.xq);
  a.xqs = reinterpret_cast<int2*>(ws + w.xqs);
  a.h = reinterpret_cast<float*>(ws + w.h);
  a.hsum = reinterpret_cast<float*>(ws + w.hsum);
  a.hq = reinterpret_cast<uint32_t*>(ws + w.hq);
  a.hqs = reinterpret_cast<int2*>(ws + w.hqs);
  a.y = reinterpret_cast<float*>(ws + w.y);
  a.wait_ns = plan->wait_ns;
  a.inject = plan->inject;
  a.idot = plan->idot;

  const bool prof = plan->prof_calls < plan->prof_max_calls;
  int launches = 0;
  auto run = [&](KernelId id, auto&& fn) -> cudaError_t {
    if (prof) {
      cudaEvent_t e0, e1;
      cudaEventCreate(&e0);
      cudaEventCreate(&e1);
      cudaEventRecord(e0, st);
      cudaError_t r = fn();
      cudaEventRecord(e1, st);
      plan->prof_events.push_back(e0);
      plan->prof_events.push_back(e1);
      plan->prof_kernel.push_back(id);
      ++launches;
      return r;
    }
    ++launches;
    return fn();
  };

  cudaError_t ce = cudaMemsetAsync(ws + w.status, 0, 64, st);
  if (ce != cudaSuccess) return cuda_fail(ce, "forward: clear status");
  if (T <= kDecodeMaxT) {
    if ((ce = run(K_ROUTE, [&] { return launch_route_decode(a, st); })) != cudaSuccess)
      return cuda_fail(ce, "forward: route_decode");
  } else {
    if (w.wsplit && router_tc_applies(a)) {   // tensor cores, fp32-exact products (router_tc.cu)
      auto encode = get_encode();
      if (!encode) return fail(COLI_ECUDA, "forward: cuTensorMapEncodeTiled is not available");
      if ((ce = run(K_RSPLIT, [&] { return launch_router_split(a, ws + w.wsplit, st); })) != cudaSuccess)
        return cuda_fail(ce, "forward: router_split");
      if ((ce = run(K_ROUTER, [&] { return launch_router_tc(a, ws + w.wsplit, encode, st); })) != cudaSuccess)
        return cuda_fail(ce, "forward: router_logits (tensor cores)");
    } else if ((ce = run(K_ROUTER, [&] { return launch_router_logits(a, st); })) != cudaSuccess) {
      return cuda_fail(ce, "forward: router_logits");
    }
    if ((ce = run(K_TOPK, [&] { return launch_router_topk(a, st); })) != cudaSuccess)
      return cuda_fail(ce, "forward: router_topk");
    if ((ce = run(K_PERMUTE, [&] { return launch_permute(a, st); })) != cudaSuccess)
      return cuda_fail(ce, "forward: permute");
  }
  if (between) {   // host step between routing and the experts (the expert cache admits the chosen experts)
    const coli_status rc = between(ctx, a, st);
    if (rc == kStopAfterRouting) {
      plan->last_launches = launches;
      return COLI_OK;
    }
    if (rc != COLI_OK) return rc;
  }
  if (T <= kDecodeMaxT) {
    if ((ce = run(K_GATEUP, [&] { return launch_decode_gateup(a, T, st, plan->num_sms); })) != cudaSuccess)
      return cuda_fail(ce, "forward: expert_gate_up");
    if ((d.qtype == COLI_Q_INT4_G128 || a.idot) &&
        (ce = run(K_PREP, [&] { return launch_quantize_h(a, st); })) != cudaSuccess)
      return cuda_fail(ce, "forward: quantize_h");
    if ((ce = run(K_DOWN, [&] { return launch_decode_down(a, T, st, plan->num_sms); })) != cudaSuccess)
      return cuda_fail(ce, "forward: expert_down");
  } else {
    // tensor-core path: fp16 activations in grouped order, tile tables, two grouped GEMMs
    const int rows = T * d.k + (d.has_shared ? T : 0);
    __half* xh = reinterpret_cast<__half*>(ws + w.xh);
    __half* hh = reinterpret_cast<__half*>(ws + w.h);
    int32_t* counts = reinterpret_cast<int32_t*>(ws + w.pf_counts);
    auto encode = get_encode();
    if (!encode) return fail(COLI_ECUDA, "forward: cuTensorMapEncodeTiled is not available");
    CUtensorMap xmap, hmap;
    {
      const cuuint64_t gdim[2] = {(cuuint64_t)d.d, (cuuint64_t)rows};
      const cuuint64_t gstr[1] = {(cuuint64_t)d.d * 2};
      const cuuint32_t box[2] = {64, (cuuint32_t)kPrefillBBox};   // 128 bytes x kPrefillBBox rows
      const cuuint32_t es[2] = {1, 1};
      CUresult r = encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xh, gdim, gstr, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(COLI_ECUDA, "forward: activation tensor map (%d)", (int)r);
      const cuuint64_t hdim[2] = {(cuuint64_t)plan->Fmax, (cuuint64_t)rows};
      const cuuint64_t hstr[1] = {(cuuint64_t)plan->Fmax * 2};
      r = encode(&hmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hh, hdim, hstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(COLI_ECUDA, "forward: hidden tensor map (%d)", (int)r);
    }
    const CUtensorMap* wmaps = tb.maps + ((size_t)tb.n_slots + 1) * 3;
    if ((ce = run(K_GATHER, [&] { return launch_gather_x(a, xh, rows, st); })) != cudaSuccess)
      return cuda_fail(ce, "forward: gather_x");
    if ((ce = run(K_TILES, [&] {
           return launch_plan_tiles(a, ws + w.chunks, ws + w.gu_tiles, ws + w.dn_tiles, counts, st);
         })) != cudaSuccess)
      return cuda_fail(ce, "forward: plan_tiles");
    if ((ce = run(K_TC_GATEUP, [&] {
           return launch_prefill_gateup(a, ws + w.chunks, ws + w.gu_tiles, counts + 1, wmaps, xmap, hh, st,
                                        plan->num_sms);
         })) != cudaSuccess)
      return cuda_fail(ce, "forward: tc_gate_up");
    if ((ce = run(K_TC_DOWN, [&] {
           return launch_prefill_down(a, ws + w.chunks, ws + w.dn_tiles, counts + 2, wmaps, hmap, a.y, st,
                                      plan->num_sms);
         })) != cudaSuccess)
      return cuda_fail(ce, "forward: tc_down");
  }
  if ((ce = run(K_COMBINE, [&] { return launch_combine(a, st); })) != cudaSuccess)
    return cuda_fail(ce, "forward: combine");
  plan->last_launches = launches;
  if (prof) plan->prof_calls++;
  return COLI_OK;
}

extern "C" {

coli_status colibri_moe_rmsnorm_bf16(const float* h, int T, int d, float eps, uint16_t* out, void* stream) {
  if (!h || !out) return fail(COLI_EINVAL, "rmsnorm: null pointer");
  if (T < 1 || d < 4 || d % 4) return fail(COLI_EINVAL, "rmsnorm: need T >= 1 and d a positive multiple of 4");
  if (!aligned(h, 16) || !aligned(out, 8)) return fail(COLI_EALIGN, "rmsnorm: h 16-byte, out 8-byte alignment");
  if (!(eps >= 0.f)) return fail(COLI_EINVAL, "rmsnorm: eps must be >= 0");
  cudaError_t ce = launch_rmsnorm_bf16(h, T, d, eps, out, static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? COLI_OK : cuda_fail(ce, "rmsnorm");
}

coli_status colibri_moe_debug_routing(const coli_moe_plan_t* plan, const void* workspace, int T, int32_t* topk_idx,
                                      float* topk_w, int32_t* near_tie, int32_t* expert_offsets, int32_t* pair_token,
                                      int32_t* pair_slot, void* stream) {
  if (!plan || !workspace) return fail(COLI_EINVAL, "debug_routing: null argument");
  if (T < 1 || T > plan->desc.T_max) return fail(COLI_EINVAL, "debug_routing: bad T");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  const WsLayout& w = plan->ws;
  const size_t k = plan->desc.k;
  struct Cp { void* dst; size_t off; size_t bytes; } cps[] = {
      {topk_idx, w.topk_idx, T * k * 4}, {topk_w, w.topk_w, T * k * 4},       {near_tie, w.near_tie, (size_t)T * 4},
      {expert_offsets, w.offsets, ((size_t)plan->desc.E + 1) * 4},            {pair_token, w.pair_token, T * k * 4},
      {pair_slot, w.pair_slot, T * k * 4}};
  for (const Cp& c : cps) {
    if (!c.dst) continue;
    cudaError_t ce = cudaMemcpyAsync(c.dst, ws + c.off, c.bytes, cudaMemcpyDefault, st);
    if (ce != cudaSuccess) return cuda_fail(ce, "debug_routing: copy");
  }
  return COLI_OK;
}

coli_status colibri_moe_check_status(const coli_moe_plan_t* plan, const void* workspace, int32_t* device_status,
                                     void* stream) {
  if (!plan || !workspace || !device_status) return fail(COLI_EINVAL, "check_status: null argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t ce =
      cudaMemcpyAsync(&v, static_cast<const uint8_t*>(workspace) + plan->ws.status, 4, cudaMemcpyDeviceToHost, st);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(st);
  if (ce != cudaSuccess) return cuda_fail(ce, "check_status");
  *device_status = v;
  if (v) return fail(COLI_EDEVICE, "device status 0x%x (bad expert id = 1, wait timeout = 2)", v);
  return COLI_OK;
}

coli_status colibri_moe_profile_begin(coli_moe_plan_t* plan, int max_calls) {
  if (!plan || max_calls < 0) return fail(COLI_EINVAL, "profile_begin: bad argument");
  for (cudaEvent_t e : plan->prof_events) cudaEventDestroy(e);
  plan->prof_events.clear();
  plan->prof_kernel.clear();
  plan->prof_calls = 0;
  plan->prof_max_calls = max_calls;
  return COLI_OK;
}

coli_status colibri_moe_profile_end(coli_moe_plan_t* plan, coli_kernel_time* out, int max_kernels, int* n_kernels) {
  if (!plan || (!out && max_kernels > 0) || !n_kernels) return fail(COLI_EINVAL, "profile_end: bad argument");
  double tot[K_COUNT] = {0};
  int cnt[K_COUNT] = {0};
  coli_status rc = COLI_OK;
  for (size_t i = 0; i < plan->prof_kernel.size(); ++i) {
    cudaEvent_t e0 = plan->prof_events[2 * i], e1 = plan->prof_events[2 * i + 1];
    float ms = 0.f;
    cudaError_t ce = cudaEventSynchronize(e1);
    if (ce == cudaSuccess) ce = cudaEventElapsedTime(&ms, e0, e1);
    if (ce != cudaSuccess && rc == COLI_OK) rc = cuda_fail(ce, "profile_end");
    tot[plan->prof_kernel[i]] += ms;
    cnt[plan->prof_kernel[i]] += 1;
  }
  int n = 0;
  for (int kid = 0; kid < K_COUNT; ++kid) {
    if (!cnt[kid]) continue;
    if (n < max_kernels) out[n] = coli_kernel_time{kKernelNames[kid], tot[kid], cnt[kid]};
    ++n;
  }
  *n_kernels = n;
  for (cudaEvent_t e : plan->prof_events) cudaEventDestroy(e);
  plan->prof_events.clear();
  plan->prof_kernel.clear();
  plan->prof_max_calls = 0;
  plan->prof_calls = 0;
  return rc;
}

int colibri_moe_last_launch_count(const coli_moe_plan_t* plan) { return plan ? plan->last_launches : 0; }

// ------------------------------------------------------------------ sparse-attention key selection

// status | scores [T][L] | counts [T] | histogram [T][65536] | coarse histogram [T][2048] |
// bitmask [T][ceil(L/32)] | candidates [T][2048] x 2   (counts and histograms adjoin: one clear covers them)
static size_t indexer_ws_bytes(int T, int L) {
  return 256 + align_up((size_t)T * (size_t)L * 4, 256);
}

coli_status colibri_indexer_workspace_size(int T_max, int L_max, size_t* bytes) {
  if (!bytes || T_max < 1 || L_max < 1) return fail(COLI_EINVAL, "indexer_workspace_size: bad argument");
  *bytes = indexer_ws_bytes(T_max, L_max);
  return COLI_OK;
}

static coli_status indexer_call(int steps, int T, int L, int pos0, int H, int d, int topk, const void* q,
                                const float* w, const void* keys, int32_t* topk_idx, void* workspace,
                                size_t workspace_bytes, void* stream) {
  if (((steps & 1) && (!q || !w || !keys)) || ((steps & 2) && !topk_idx) || !workspace)
    return fail(COLI_EINVAL, "indexer_topk: null pointer");
  if (T < 1 || L < 1 || topk < 1 || pos0 < 0) return fail(COLI_EINVAL, "indexer_topk: need T, L, topk >= 1, pos0 >= 0");
  if (H != 64 || d != 128)
    return fail(COLI_EUNSUPPORTED, "indexer_topk: this build serves 64 heads of 128 (got %d x %d)", H, d);
  if ((long long)T * L > (1LL << 31)) return fail(COLI_EUNSUPPORTED, "indexer_topk: T*L too large");
  if (L > (1 << 17)) return fail(COLI_EUNSUPPORTED, "indexer_topk: this build selects among at most 131072 keys");
  if (workspace_bytes < indexer_ws_bytes(T, L))
    return fail(COLI_EWORKSPACE, "indexer_topk: workspace %zu bytes < required %zu", workspace_bytes,
                indexer_ws_bytes(T, L));
  if (!aligned(workspace, 256)) return fail(COLI_EALIGN, "indexer_topk: workspace not 256-byte aligned");
  if (((steps & 1) && (!aligned(q, 16) || !aligned(keys, 16) || !aligned(w, 4))) ||
      ((steps & 2) && !aligned(topk_idx, 4)))
    return fail(COLI_EALIGN, "indexer_topk: q and keys 16-byte, w and topk_idx 4-byte alignment");
  auto encode = get_encode();
  if (!encode) return fail(COLI_ECUDA, "indexer_topk: cuTensorMapEncodeTiled is not available");
  int dev = 0, sms = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (ce != cudaSuccess) return cuda_fail(ce, "indexer_topk: device query");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (steps & 1) {
    ce = cudaMemsetAsync(ws, 0, 64, st);
    if (ce != cudaSuccess) return cuda_fail(ce, "indexer_topk: clear status");
  }
  IndexerCall c;
  c.T = T;
  c.L = L;
  c.pos0 = pos0;
  c.topk = topk;
  c.q = q;
  c.w = w;
  c.keys = keys;
  c.scores = reinterpret_cast<float*>(ws + 256);
  c.out = topk_idx;
  c.status = reinterpret_cast<int32_t*>(ws);
  c.wait_ns = kWaitLimitNs;
  c.encode = encode;
  c.steps = steps;
  ce = launch_indexer(c, st, sms);
  return ce == cudaSuccess ? COLI_OK : cuda_fail(ce, "indexer_topk: launch");
}

coli_status colibri_indexer_topk(int T, int L, int pos0, int H, int d, int topk, const void* q, const float* w,
                                 const void* keys, int32_t* topk_idx, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  return indexer_call(3, T, L, pos0, H, d, topk, q, w, keys, topk_idx, workspace, workspace_bytes, stream);
}

coli_status colibri_indexer_scores(int T, int L, int pos0, int H, int d, const void* q, const float* w,
                                   const void* keys, void* workspace, size_t workspace_bytes, void* stream) {
  return indexer_call(1, T, L, pos0, H, d, 1, q, w, keys, nullptr, workspace, workspace_bytes, stream);
}

coli_status colibri_indexer_select(int T, int L, int pos0, int topk, int32_t* topk_idx, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  return indexer_call(2, T, L, pos0, 64, 128, topk, nullptr, nullptr, nullptr, topk_idx, workspace,
                      workspace_bytes, stream);
}

coli_status colibri_indexer_check_status(const void* workspace, int32_t* device_status, void* stream) {
  if (!workspace || !device_status) return fail(COLI_EINVAL, "indexer_check_status: null argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t ce = cudaMemcpyAsync(&v, workspace, 4, cudaMemcpyDeviceToHost, st);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(st);
  if (ce != cudaSuccess) return cuda_fail(ce, "indexer_check_status");
  *device_status = v;
  if (v) return fail(COLI_EDEVICE, "indexer device status 0x%x (wait timeout = 2)", v);
  return COLI_OK;
}

coli_status colibri_moe_debug_hidden(const coli_moe_plan_t* plan, const void* workspace, int T, float* h_out,
                                     void* stream) {
  if (!plan || !workspace || !h_out) return fail(COLI_EINVAL, "debug_hidden: null argument");
  if (T < 1 || T > plan->desc.T_max) return fail(COLI_EINVAL, "debug_hidden: bad T");
  if (!aligned(h_out, 4)) return fail(COLI_EALIGN, "debug_hidden: h_out must be 4-byte aligned");
  const coli_moe_desc& d = plan->desc;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  const WsLayout& w = plan->ws;
  HiddenView v;
  const bool i4 = d.qtype == COLI_Q_INT4_G128;
  if (T > kDecodeMaxT) v.mode = 4;
  else if (plan->idot) v.mode = i4 ? 2 : 3;
  else v.mode = i4 ? 0 : 1;
  v.perm = i4 ? 1 : 0;
  v.qtype = d.qtype;
  v.P = T * d.k;
  v.rows = v.P + (d.has_shared ? T : 0);
  v.F = d.d_ff;
  v.Fs = d.has_shared ? d.shared_d_ff : 0;
  v.Fmax = plan->Fmax;
  v.h = reinterpret_cast<const float*>(ws + w.h);
  v.hq = ws + w.hq;
  v.hqs = reinterpret_cast<const int2*>(ws + w.hqs);
  v.hh = reinterpret_cast<const __half*>(ws + w.h);
  v.out = h_out;
  const cudaError_t ce = launch_debug_hidden(v, static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? COLI_OK : cuda_fail(ce, "debug_hidden");
}

coli_status colibri_moe_set_idot(coli_moe_plan_t* plan, int enable) {
  if (!plan) return fail(COLI_EINVAL, "set_idot: null plan");
  if (enable != 0 && enable != 1) return fail(COLI_EINVAL, "set_idot: enable must be 0 or 1, got %d", enable);
  plan->idot = enable;
  return COLI_OK;
}

coli_status colibri_moe_debug_inject(coli_moe_plan_t* plan, int flags, double wait_limit_ms) {
  if (!plan) return fail(COLI_EINVAL, "debug_inject: null plan");
  if (flags & ~(COLI_INJECT_WITHHOLD_STAGE | COLI_INJECT_BAD_EXPERT_ID))
    return fail(COLI_EINVAL, "debug_inject: unknown flag bits 0x%x", flags);
  if (!(wait_limit_ms == wait_limit_ms)) return fail(COLI_EINVAL, "debug_inject: wait limit is NaN");
  plan->inject = flags;
  plan->wait_ns = wait_limit_ms > 0 ? (unsigned long long)(wait_limit_ms * 1e6) : kWaitLimitNs;
  if (plan->wait_ns < 1000) plan->wait_ns = 1000;
  return COLI_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ forward without caller workspace
//
// For callers that cannot allocate device memory at all: code running under a
// host framework that owns every allocation, or inside a region where an
// allocation is not allowed.  The workspace of the forward pass lives in a
// fixed file-scope device array instead.  Its address is a device address
// only when taken with cudaGetSymbolAddress on the device that uses it (the
// array's name in host code is a host-side stand-in), so the first call on
// each device looks it up once and caches it.

namespace {
constexpr size_t kNoAllocScratchBytes = 8u << 20;   // 8 MiB, held by every device that loads the library
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
constexpr int kNoAllocMaxDevices = 64;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {nullptr};
std::mutex g_noalloc_mu;
}  // namespace

extern "C" coli_status colibri_moe_forward_noalloc(const coli_moe_plan_t* plan, int T, const void* x,
                                                   const float* router_w, const float* bias, const float* residual,
                                                   float* out, void* stream) {
  if (!plan) return fail(COLI_EINVAL, "forward_noalloc: null plan");
  if (plan->ws.total > kNoAllocScratchBytes)
    return fail(COLI_EWORKSPACE,
                "forward_noalloc: this plan needs %zu bytes of workspace, more than the %zu-byte static scratch; "
                "use a smaller T_max or colibri_moe_forward with a caller workspace",
                plan->ws.total, kNoAllocScratchBytes);
  if (plan->prof_calls < plan->prof_max_calls)
    return fail(COLI_ESTATE, "forward_noalloc: per-kernel profiling is active on this plan (it creates events)");
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce, "forward_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(COLI_EUNSUPPORTED, "forward_noalloc: device index %d", dev);
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      ce = cudaGetSymbolAddress(&g_noalloc_ptr[dev], g_noalloc_scratch);
      if (ce != cudaSuccess) {
        g_noalloc_ptr[dev] = nullptr;
        return cuda_fail(ce, "forward_noalloc: cudaGetSymbolAddress(scratch)");
      }
    }
    scratch = g_noalloc_ptr[dev];
  }
  return colibri_moe_forward(plan, T, x, router_w, bias, residual, out, scratch, kNoAllocScratchBytes, stream);
}
