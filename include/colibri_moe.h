/*
 * colibri_moe.h -- C ABI of a quantized sparse Mixture-of-Experts layer
 * forward for one NVIDIA GB300 GPU (sm_103a).
 *
 * The layer (the MoE hot path of the Colibri engine):
 *   1. router: logits z = x Wr^T, s = sigmoid(z), u = s + bias; the k experts
 *      with the largest u are chosen ("25GB RAM runs 744B GLM-5.2" page
 *      (pwwt.cn), section 3.1: DeepSeek-V3 style sigmoid router, 8 of 256
 *      experts per token; section 4.3: the expert bias of auxiliary-loss-free
 *      balancing steers selection).  Ties go to the lower expert id.
 *   2. gate weights g = routed_scale * s / sum(s over the chosen experts).
 *   3. batch-union grouping (same page, section 3.4): (token, slot) pairs are
 *      grouped by expert, so each chosen expert's weights are streamed once
 *      for all of its tokens.
 *   4. per-expert SwiGLU FFN y = Wd (silu(Wg x) * (Wu x)) on int4 / int8
 *      weights with per-output-channel scale and zero-point ("Colibri
 *      walkthrough" page (discosf.com), section 3.4): w = (q - zp) * scale.
 *   5. optional always-on shared expert ("25GB RAM" page, section 2), weight 1.
 *   6. out[t] = residual[t] + sum_j g[t][j] * y[t][j] + y_shared[t].
 *
 * Conventions for every call:
 *   - Pointers named "device" are CUDA device (or managed) pointers of the
 *     current device; "host" pointers are ordinary CPU memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls that take a stream are asynchronous on it and never
 *     synchronise the host.
 *   - Errors are returned as coli_status; nothing aborts or throws.  The
 *     message of the last error on the calling thread is returned by
 *     colibri_moe_last_error().  Argument checks happen before any launch.
 *   - The caller owns every tensor and the workspace.  A plan owns only its
 *     host metadata and a small device table of expert descriptors that it
 *     frees in colibri_moe_destroy().
 */
#ifndef COLIBRI_MOE_H
#define COLIBRI_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* exported symbols of the shared library */
#if defined(__GNUC__)
#define COLI_API __attribute__((visibility("default")))
#else
#define COLI_API
#endif

typedef enum {
  COLI_OK = 0,
  COLI_EINVAL = 1,          /* bad shape, null pointer, T out of range */
  COLI_EALIGN = 2,          /* a pointer is not aligned as documented */
  COLI_EUNSUPPORTED = 3,    /* valid request this build cannot serve (qtype, sizes) */
  COLI_EWORKSPACE = 4,      /* workspace smaller than colibri_moe_plan reported */
  COLI_ECUDA = 5,           /* a CUDA runtime call failed (message has the CUDA error) */
  COLI_EDEVICE = 6,         /* a kernel reported an error in the workspace status word */
  COLI_ESTATE = 7           /* call out of order (e.g. forward before bind) */
} coli_status;

typedef enum {
  /* int4 codes, groups of 128 consecutive inputs of one output row share an
     fp16 scale and a 4-bit zero-point */
  COLI_Q_INT4_G128 = 0,
  /* int8 codes, one fp32 scale and one 8-bit zero-point per output row */
  COLI_Q_INT8_PC = 1
} coli_qtype;

typedef enum { COLI_X_BF16 = 0, COLI_X_F32 = 1 } coli_xtype;

/*
 * One quantised matrix W[N][K] (N output rows, K inputs), device pointers.
 *   COLI_Q_INT4_G128: q     uint8 [N][K/2], byte j of a row holds inputs 2j
 *                           (low nibble) and 2j+1 (high nibble);
 *                     scale fp16 [N][K/128];
 *                     zp    uint8 [N][ceil(K/256)], low nibble = even group.
 *   COLI_Q_INT8_PC:   q     uint8 [N][K]; scale float [N]; zp uint8 [N].
 * Dequantised weight: (code - zero_point) * scale.
 * q must be 16-byte aligned (it is streamed with TMA); scale and zp need only
 * their element alignment.
 */
typedef struct {
  const void* q;
  const void* scale;
  const void* zp;
} coli_qmat;

/* One expert: gate and up are [d_ff][d], down is [d][d_ff]. */
typedef struct {
  coli_qmat gate, up, down;
} coli_expert;

/*
 * Layer description.
 *   T_max       largest token count a forward call may pass (>= 1).
 *   d           hidden size; d_ff the routed experts' FFN size.
 *   E, k        number of routed experts and experts chosen per token
 *               (1 <= k <= min(E, 32), E <= 1024).
 *   routed_scale the factor applied to the renormalised gate weights.
 *   qtype       coli_qtype of every expert matrix (shared expert included).
 *   xtype       coli_xtype of x.
 *   has_shared  1 = one always-on shared expert with FFN size shared_d_ff.
 * Sizes supported by the kernels: d and the FFN sizes are multiples of 256
 * (int4) or 128 (int8).
 */
typedef struct {
  int T_max;
  int d;
  int d_ff;
  int E;
  int k;
  float routed_scale;
  int qtype;
  int xtype;
  int has_shared;
  int shared_d_ff;
} coli_moe_desc;

typedef struct coli_moe_plan coli_moe_plan_t;

/*
 * Validate `desc` and create a plan (host memory only; no CUDA call).
 * The description fixes the layer of the "25GB RAM runs 744B GLM-5.2" page:
 * E routed experts of which k are chosen per token (section 3.1), int4 or
 * int8 weights with per-channel scale and zero point ("Colibri walkthrough"
 * page, section 3.4), an optional resident shared expert (section 2).  The
 * workspace holds the batch-union grouping of section 3.4: per-expert pair
 * lists, so that each chosen expert is streamed once for all its tokens.
 * *workspace_bytes receives the size of the device workspace a forward call
 * needs for up to T_max tokens (256-byte aligned base required).
 * Errors: COLI_EINVAL (null argument, bad sizes), COLI_EUNSUPPORTED.
 */
COLI_API coli_status colibri_moe_plan(const coli_moe_desc* desc, coli_moe_plan_t** plan, size_t* workspace_bytes);

/*
 * Bind the expert weights (the resident "expert slots" of the "Colibri
 * walkthrough" page, section 3.1; here every expert of the layer is resident
 * in device memory, one contiguous block per expert matrix as in its
 * section 4.2 layout) to a plan on the
 * current device.  experts: HOST array [E] of descriptors holding device
 * pointers; shared: HOST pointer to one descriptor, or NULL when the plan has
 * no shared expert.  The weights themselves are not copied: they must stay
 * allocated and unchanged while the plan is used.  Synchronous: builds the
 * TMA tensor maps and uploads the descriptor table (plan-owned device memory,
 * freed by colibri_moe_destroy).  May be called again to rebind.
 * Errors: COLI_EINVAL (null pointer), COLI_EALIGN (q not 16-byte aligned),
 * COLI_ECUDA.
 */
COLI_API coli_status colibri_moe_bind_experts(coli_moe_plan_t* plan, const coli_expert* experts, const coli_expert* shared);

/*
 * One layer forward for T tokens (1 <= T <= T_max), asynchronous on stream:
 * steps 1-6 at the top of this header ("25GB RAM runs 744B GLM-5.2" page,
 * sections 3.1, 3.4 and 4.3; "Colibri walkthrough" page, section 3.4).
 *   x         device [T][d], bf16 or fp32 per desc.xtype (16-byte aligned).
 *   router_w  device float [E][d] (16-byte aligned).
 *   bias      device float [E]: selection-only router bias.
 *   residual  device float [T][d] added to the output, or NULL.  May equal out.
 *   out       device float [T][d].
 *   workspace device, >= the size colibri_moe_plan reported, 256-byte aligned.
 * Two calls that overlap on the GPU need two workspaces.
 * Errors: COLI_EINVAL, COLI_EALIGN, COLI_EWORKSPACE, COLI_ESTATE (not bound),
 * COLI_ECUDA (launch failure).
 */
COLI_API coli_status colibri_moe_forward(const coli_moe_plan_t* plan, int T, const void* x, const float* router_w,
                                const float* bias, const float* residual, float* out, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * The same forward pass with no workspace argument, for callers that cannot
 * allocate device memory (a host framework that owns all allocations, or a
 * region of code where allocating is not allowed).  There is no counterpart
 * in the pages; this is an interface convenience.
 *   The workspace is a fixed 8 MiB array in the library's device memory (every
 *   GPU that loads the library holds it until the process exits).  Plans whose
 *   workspace (colibri_moe_plan's *workspace_bytes) exceeds 8 MiB are refused
 *   with COLI_EWORKSPACE; that covers decode-sized plans (GLM-class layer:
 *   T_max up to about 16).
 *   The first call on a device looks up the array's device address once
 *   (cudaGetSymbolAddress) and caches it; make that first call before any
 *   stream capture.  Nothing is allocated (no cudaMalloc or cudaFree).
 *   Every call on a device shares the one array and leaves its contents
 *   behind; each call clears what must start at zero.  Calls that overlap on
 *   the GPU (different streams, or different host threads) race on the array
 *   and must be serialised by the caller.  Refused (COLI_ESTATE) while
 *   per-kernel profiling is active on the plan.
 * Other arguments and errors as colibri_moe_forward.
 */
COLI_API coli_status colibri_moe_forward_noalloc(const coli_moe_plan_t* plan, int T, const void* x,
                                                 const float* router_w, const float* bias, const float* residual,
                                                 float* out, void* stream);

/*
 * RMSNorm with unit gain, rounded to bf16 (the input of the next stacked
 * layer): out[t][i] = bf16(h[t][i] / sqrt(mean_i(h[t][i]^2) + eps)).
 * h device float [T][d]; out device uint16 (bf16 bits) [T][d]; d % 4 == 0.
 */
COLI_API coli_status colibri_moe_rmsnorm_bf16(const float* h, int T, int d, float eps, uint16_t* out, void* stream);

/*
 * Routing check (the pages ask for exact routing: "25GB RAM runs 744B
 * GLM-5.2" page, section 4.3, DeepSeek-V3 sigmoid router, selection and
 * scaling).  Copy the routing state of the last forward that used `workspace` into
 * caller buffers (device pointers, any may be NULL), asynchronously on stream:
 *   topk_idx int32 [T][k]  chosen experts, ascending ids per token
 *   topk_w   float [T][k]  gate weights in the same order
 *   near_tie int32 [T]     1 where the k-th and (k+1)-th selection scores
 *                          differ by less than 1e-5
 *   expert_offsets int32 [E+1]  start of each expert's pairs in grouped order
 *   pair_token, pair_slot int32 [T*k]  (token, slot) of each grouped pair,
 *                          sorted by (expert, token, slot)
 * Errors: COLI_EINVAL, COLI_ECUDA.
 */
COLI_API coli_status colibri_moe_debug_routing(const coli_moe_plan_t* plan, const void* workspace, int T, int32_t* topk_idx,
                                      float* topk_w, int32_t* near_tie, int32_t* expert_offsets, int32_t* pair_token,
                                      int32_t* pair_slot, void* stream);

/*
 * Read the device status word of `workspace` (synchronises `stream`).
 * *device_status = 0 when the last forward ran clean; otherwise a bit set of
 * COLI_DEV_* flags.  Returns COLI_EDEVICE when the word is non-zero.
 */
#define COLI_DEV_BAD_EXPERT_ID 1   /* a router index outside [0, E) reached the grouping step */
#define COLI_DEV_WAIT_TIMEOUT 2    /* a pipeline wait gave up after its time limit (~1 s) */
#define COLI_DEV_SELECT_ROUNDS 4   /* the key selection's rounds did not narrow to one value (not expected) */
COLI_API coli_status colibri_moe_check_status(const coli_moe_plan_t* plan, const void* workspace, int32_t* device_status,
                                     void* stream);

/*
 * Failure-path testing (no counterpart in the pages: it exercises the
 * bounded waits and the expert-id check above).  Makes the following forward
 * calls of this plan:
 *   COLI_INJECT_WITHHOLD_STAGE  skip the TMA issue of one pipeline stage of the
 *                               gate/up expert kernel (the first stage of warp 0
 *                               of CTA 0 at decode, of CTA 0 at prefill), so
 *                               that the roles waiting on it reach the wait
 *                               limit, record COLI_DEV_WAIT_TIMEOUT, drain what
 *                               they issued, free tensor memory and return;
 *   COLI_INJECT_BAD_EXPERT_ID   replace the first chosen expert id of token 0
 *                               by -1 before grouping, so that the grouping step
 *                               records COLI_DEV_BAD_EXPERT_ID and leaves that
 *                               pair out of the output.
 * Nothing faults or hangs: every wait stays bounded.  wait_limit_ms > 0 sets
 * the limit of every pipeline wait (default ~1000 ms); <= 0 restores it.
 * flags = 0 turns injection off.  The outputs of an injected forward are not
 * meaningful; the next forward without injection is a normal one.
 * Errors: COLI_EINVAL (null plan or unknown flag bits).
 */
/*
 * Integer-dot expert inputs (the IDOT switch of the "25GB RAM runs 744B
 * GLM-5.2" page, section 6 (reproducibility): integer kernels whose rounding
 * depends on the batch shape, so that their output may differ slightly from
 * the single-token path).  enable = 1: the inputs of the expert matrices (x for
 * gate and up, the SwiGLU output h for down) are cut into blocks of 32 values
 * that share the scale 2^(e-6), e = floor(log2(max |v|)) over the block (at
 * least -100), and each value becomes the int8 code round-half-even(v / 2^(e-6))
 * clamped to [-127, 127].  Up to 8 tokens per call the expert kernels take
 * integer dot products of the weight codes with these codes; above that the
 * tensor-core kernels take the values code * 2^(e-6) as fp16 operands, which is
 * exact for 2^-18 <= max |v| < 2^16 per block.  Routing always reads x itself.
 * enable = 0 (the default) restores the default inputs.  Takes effect at the
 * next forward call.  Errors: COLI_EINVAL (null plan, enable not 0 or 1).
 */
COLI_API coli_status colibri_moe_set_idot(coli_moe_plan_t* plan, int enable);

/*
 * Test and debugging aid: the input of the down projection in the last
 * forward call on `workspace` (made with T tokens and the plan's current IDOT
 * setting), as the down kernels read it (the SwiGLU output h of the "Colibri
 * walkthrough" page, section 3.4, after the kernels' own conversion: 16-bit
 * fixed point, integer-dot codes times their block scale, or fp16).
 * h_out: DEVICE memory, [T*k + (has_shared ? T : 0)][max(d_ff, shared_d_ff)]
 * floats; rows in the grouped order of colibri_moe_debug_routing's pair_token
 * and pair_slot, then the shared expert's rows (token order); columns past the
 * row's expert's FFN size are 0.  Asynchronous on `stream`.
 * Errors: COLI_EINVAL (null argument, bad T), COLI_EALIGN, COLI_ECUDA.
 */
COLI_API coli_status colibri_moe_debug_hidden(const coli_moe_plan_t* plan, const void* workspace, int T,
                                              float* h_out, void* stream);

#define COLI_INJECT_WITHHOLD_STAGE 1
#define COLI_INJECT_BAD_EXPERT_ID 2
COLI_API coli_status colibri_moe_debug_inject(coli_moe_plan_t* plan, int flags, double wait_limit_ms);

/*
 * Per-kernel timing (the per-stage share that a "--profile" run reports).
 * colibri_moe_profile_begin(plan, max_calls) makes the next forward calls
 * record a CUDA event before and after every kernel, on the launching stream,
 * for up to max_calls calls.  colibri_moe_profile_end() synchronises those
 * events, writes up to max_kernels entries of {name, total ms, launches}
 * (names are static strings owned by the library) and returns the number of
 * distinct kernels in *n_kernels; profiling is then off.
 */
typedef struct {
  const char* name;
  double total_ms;
  int launches;
} coli_kernel_time;
COLI_API coli_status colibri_moe_profile_begin(coli_moe_plan_t* plan, int max_calls);
COLI_API coli_status colibri_moe_profile_end(coli_moe_plan_t* plan, coli_kernel_time* out, int max_kernels, int* n_kernels);

/*
 * Expert-slot cache in device memory with a host-memory tier.
 * "25GB RAM runs 744B GLM-5.2" page, section 2: the weights are spread over a
 * hierarchy of storage tiers and the routed experts a layer needs are read on
 * demand; section 3.5: a per-layer LRU cache of experts, the next experts read
 * ahead asynchronously.  "Colibri walkthrough" page, section 3.1: one "expert
 * slot" holds one expert's weights; a slot keeps last_used and hit_count and
 * eviction prefers a low hit_count and an old last_used; the engine reports
 * cache_hit_rate.  Here the lower tier is host memory and the upper tier a
 * pool of slots in device memory (one cache per layer).
 *
 * colibri_moe_cache_slot_bytes: device bytes of one slot (one packed expert).
 * colibri_moe_cache_create: n_slots slots in caller-owned device memory
 *   slot_memory (>= n_slots * slot bytes, 256-byte aligned, kept while the
 *   cache lives); host_experts: HOST array [E] of descriptors whose pointers
 *   are host memory (pinned memory makes the copies asynchronous and fast)
 *   holding every routed expert in the layout of coli_qmat (an expert whose
 *   nine arrays sit at the offsets of the slot layout -- 256-byte aligned, in
 *   the order gate q, scale, zp, up ..., down ... -- moves in one copy); shared: device
 *   descriptor of the resident shared expert (or NULL).  weight >= 0: the
 *   eviction weighting -- the victim is the slot, unused by the current
 *   forward, with the smallest last_used + weight * hit_count (hit_count =
 *   forwards that used the expert since it entered the slot; 0 = plain LRU;
 *   ties to the older last_used, then the lower slot).  Allocates the cache's
 *   small device tables.  Errors: COLI_EINVAL, COLI_EALIGN, COLI_EWORKSPACE,
 *   COLI_ECUDA.
 * colibri_moe_forward_cached: the layer forward with weights from the cache.
 *   After the routing kernels it reads the chosen experts back (it
 *   synchronises `stream` once), copies each missing expert into a victim slot
 *   (cudaMemcpyAsync on `stream`) and runs the expert kernels on the slots:
 *   the output equals colibri_moe_forward's exactly.  Other arguments as
 *   colibri_moe_forward; COLI_EUNSUPPORTED if the forward needs more distinct
 *   experts than there are slots.
 * colibri_moe_cache_prefetch: load the given experts (host array of ids) ahead
 *   of use on `stream` (e.g. the next layer's predicted experts).  It must not
 *   run while a forward of the same cache reads the slots on another stream:
 *   order `stream` after such forwards (an event), and the next forward after
 *   the prefetch copies.
 * colibri_moe_cache_stats / _reset_stats: counters since creation or reset
 *   (cache_hit_rate = hits / lookups).
 * colibri_moe_cache_resident: HOST array [E] receives each expert's slot or -1.
 * colibri_moe_cache_simulate: host only, no GPU: the same policy over a trace
 *   of n_steps forwards (expert_sets: the distinct ids of each step, set_sizes
 *   their counts) -> total hits and misses; for choosing n_slots and weight.
 */
typedef struct coli_cache coli_cache_t;
typedef struct {
  long long forwards;
  long long lookups;      /* experts the forwards needed */
  long long hits;
  long long misses;
  long long evictions;
  long long prefetched;   /* experts loaded by colibri_moe_cache_prefetch */
  long long bytes_copied; /* host -> device */
  long long predicted;    /* experts named by colibri_moe_cache_pilot */
} coli_cache_stats;
COLI_API coli_status colibri_moe_cache_slot_bytes(const coli_moe_plan_t* plan, size_t* bytes);
COLI_API coli_status colibri_moe_cache_create(coli_moe_plan_t* plan, int n_slots, double weight,
                                              const coli_expert* host_experts, const coli_expert* shared,
                                              void* slot_memory, size_t slot_memory_bytes, coli_cache_t** cache);
COLI_API coli_status colibri_moe_forward_cached(coli_moe_plan_t* plan, coli_cache_t* cache, int T, const void* x,
                                                const float* router_w, const float* bias, const float* residual,
                                                float* out, void* workspace, size_t workspace_bytes, void* stream);
COLI_API coli_status colibri_moe_cache_prefetch(coli_cache_t* cache, const int32_t* experts, int n, void* stream);
COLI_API coli_status colibri_moe_cache_stats(const coli_cache_t* cache, coli_cache_stats* stats);
COLI_API coli_status colibri_moe_cache_reset_stats(coli_cache_t* cache);
COLI_API coli_status colibri_moe_cache_resident(const coli_cache_t* cache, int32_t* slot_of_expert);
COLI_API void colibri_moe_cache_destroy(coli_cache_t* cache);
/*
 * Next-layer routing prediction with read-ahead ("25GB RAM runs 744B GLM-5.2"
 * page, section 3.5: the experimental PILOT mode predicts the next layer's
 * routing from the current layer's state and reads those experts ahead).
 * Runs the next layer's router (plan_next, router_w, bias) on x -- the current
 * layer's input state, in the next layer's input type -- reads the chosen
 * experts back (it synchronises `stream` once) and prefetches them into
 * cache_next on `stream` (up to its slot count).  predicted (HOST int32
 * [min(E, T*k)], may be NULL) and *n_predicted receive the predicted experts
 * in ascending order.  workspace: a workspace of plan_next that no running
 * forward uses.  Use a stream other than the current layer's so that the
 * copies overlap its compute; as with colibri_moe_cache_prefetch, `stream`
 * must be ordered after every earlier forward of cache_next that may still
 * read its slots (e.g. wait on an event recorded after that forward), and the
 * next forward of cache_next must wait for the prefetch copies.  Errors as
 * colibri_moe_forward and colibri_moe_cache_prefetch.
 */
COLI_API coli_status colibri_moe_cache_pilot(coli_moe_plan_t* plan_next, coli_cache_t* cache_next, int T, const void* x,
                                             const float* router_w, const float* bias, int32_t* predicted,
                                             int* n_predicted, void* workspace, size_t workspace_bytes, void* stream);
COLI_API coli_status colibri_moe_cache_simulate(int E, int n_slots, double weight, const int32_t* expert_sets,
                                                const int32_t* set_sizes, int n_steps, int64_t* hits,
                                                int64_t* misses);

/*
 * Key selection of sparse attention (DSA "lightning indexer" and top-k):
 * "25GB RAM runs 744B GLM-5.2" page, section 3.3: each layer keeps only the
 * top-2048 causal keys for attention; section 4.4: a light indexer scores the
 * earlier keys, then the top-k entries are selected.  The pages give no
 * scoring formula; this library computes that of the DeepSeek-V3.2 indexer
 * the page cites:
 *   I[t][s] = sum_{j < H} w[t][j] * relu(q[t][j] . k[s]),
 * for the keys s <= pos0 + t (and s < L) that query t, at position pos0 + t,
 * sees; the topk largest are kept, a tie going to the lower key index.
 *   q        device bf16 [T][H][d] (16-byte aligned); w device float [T][H];
 *   keys     device bf16 [L][d] (16-byte aligned);
 *   topk_idx device int32 [T][topk]: the selected keys in ascending order,
 *            -1 padded when a query sees fewer than topk keys.
 *   workspace device, >= colibri_indexer_workspace_size(T, L) bytes, 256-byte
 *            aligned.  Layout: int32 status word at offset 0; the fp32 scores
 *            [T][L] at offset 256 (-infinity where a key is not visible).
 * This build serves H = 64 heads of d = 128 and L <= 131072 keys
 * (COLI_EUNSUPPORTED otherwise).
 * Asynchronous on stream; errors: COLI_EINVAL, COLI_EALIGN, COLI_EWORKSPACE,
 * COLI_EUNSUPPORTED, COLI_ECUDA.  colibri_indexer_check_status reads the
 * status word (COLI_DEV_WAIT_TIMEOUT if a pipeline wait gave up,
 * COLI_DEV_SELECT_ROUNDS if the selection did not converge).
 */
COLI_API coli_status colibri_indexer_workspace_size(int T_max, int L_max, size_t* bytes);
COLI_API coli_status colibri_indexer_topk(int T, int L, int pos0, int H, int d, int topk, const void* q, const float* w,
                                          const void* keys, int32_t* topk_idx, void* workspace, size_t workspace_bytes,
                                          void* stream);
COLI_API coli_status colibri_indexer_check_status(const void* workspace, int32_t* device_status, void* stream);
/* The two steps of colibri_indexer_topk on their own (same arguments and
 * workspace): the scores into the workspace, then the selection from them. */
COLI_API coli_status colibri_indexer_scores(int T, int L, int pos0, int H, int d, const void* q, const float* w,
                                            const void* keys, void* workspace, size_t workspace_bytes, void* stream);
COLI_API coli_status colibri_indexer_select(int T, int L, int pos0, int topk, int32_t* topk_idx, void* workspace,
                                            size_t workspace_bytes, void* stream);

/* Number of kernel launches the last forward call of this plan issued. */
COLI_API int colibri_moe_last_launch_count(const coli_moe_plan_t* plan);

/* Message of the last error returned on the calling thread ("" if none). */
COLI_API const char* colibri_moe_last_error(void);

/* Free a plan and its device descriptor table.  NULL is ignored. */
COLI_API void colibri_moe_destroy(coli_moe_plan_t* plan);

#ifdef __cplusplus
}
#endif
#endif /* COLIBRI_MOE_H */
