// Internal host-side definitions shared by the C-ABI files (api.cu, cache.cu):
// the plan object, error reporting, tensor-map encoding of one expert, and
// the forward launch sequence with a hook between routing and the experts.
#pragma once

#include <vector>

#include "moe_internal.cuh"

namespace coli {

coli_status fail(coli_status s, const char* fmt, ...);
coli_status cuda_fail(cudaError_t e, const char* what);
PFN_cuTensorMapEncodeTiled_v12000 get_encode();

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Descriptor and TMA maps of one expert whose three matrices are at the device
// pointers of `ex`: dec[3] (dequant-GEMV boxes) and tc[3] (tensor-core boxes).
coli_status encode_expert(const coli_moe_desc& d, int F, const coli_expert& ex, int id, DevExpert& dx,
                          CUtensorMap* dec, CUtensorMap* tc);

// Where the expert kernels read weights: n_slots + 1 descriptors (the last one:
// the shared expert), their maps, and the expert -> slot table (NULL: identity).
struct ExpertTables {
  const DevExpert* experts;
  const CUtensorMap* maps;
  int n_slots;
  const int32_t* slot_of;
};

// Called between the routing kernels and the expert kernels of a forward (after
// the routing is launched on `st`); returns COLI_OK to go on, kStopAfterRouting
// to end the call there (a routing-only pass), or an error.
typedef coli_status (*BetweenFn)(void* ctx, const FwdArgs& a, cudaStream_t st);
constexpr coli_status kStopAfterRouting = static_cast<coli_status>(100);

}  // namespace coli

struct coli_moe_plan {
  coli_moe_desc desc;
  coli::WsLayout ws;
  int Fmax;
  bool bound = false;
  int device = -1;
  int num_sms = 0;
  coli::DevExpert* d_experts = nullptr;
  CUtensorMap* d_maps = nullptr;
  // profiling
  int prof_max_calls = 0;
  int prof_calls = 0;
  std::vector<cudaEvent_t> prof_events;  // 2 per kernel launch
  std::vector<int> prof_kernel;          // kernel id per event pair
  int last_launches = 0;
  // failure-path testing (colibri_moe_debug_inject)
  int inject = 0;
  // integer-dot expert inputs (colibri_moe_set_idot)
  int idot = 0;
  unsigned long long wait_ns = coli::kWaitLimitNs;
};

namespace coli {
coli_status forward_impl(coli_moe_plan* plan, const ExpertTables& tb, BetweenFn between, void* ctx, int T,
                         const void* x, const float* router_w, const float* bias, const float* residual, float* out,
                         void* workspace, size_t workspace_bytes, void* stream);
}  // namespace coli
