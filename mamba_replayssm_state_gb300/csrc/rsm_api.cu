// rsm_api.cu -- host side of libreplayssm.so: argument validation, choice of
// the compiled kernel instance, launch sizing and the launch itself.
//
// The checks follow the flashinfer.mamba.replayssm_materialize API page
// (Parameters: heads_per_group divides num_heads, max_window range, one-byte
// state needs dim=64/dstate=128, BF16 inputs, a seed when philox_rounds > 0)
// and FlashInfer PR #4815's review fixes (num_heads must fit a 32-bit int;
// the thread count is a compile-time 32-wide warp multiple).  Nothing here
// reads device memory, allocates or synchronizes.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>

#include "../../include/replayssm.h"
#include "gdn_params.h"
#include "rsm_instances.h"
#include "rsm_params.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

struct Instance {
  int sf, inf, dim, dstate;
  const void* (*kernel)();     // philox_rounds == 0 (16-bit and fp32 state: every call)
  const void* (*kernel_sr)();  // one-byte state with philox_rounds > 0; NULL otherwise
};

template <int SF, int IF, int D, int N>
constexpr const void* (*sr_kernel_getter())() {
  if constexpr (SF == RSM_I8 || SF == RSM_FP8_E4M3)
    return &rsm::kernel_for_sr<SF, IF, D, N>;
  else
    return nullptr;
}

#define RSM_ENTRY(SF, IF, D, N) {SF, IF, D, N, &rsm::kernel_for<SF, IF, D, N>, sr_kernel_getter<SF, IF, D, N>()},
const Instance kInstances[] = {RSM_FOR_EACH_INSTANCE(RSM_ENTRY)};
#undef RSM_ENTRY

int elem_bytes(int dt) {
  switch (dt) {
    case RSM_F32: return 4;
    case RSM_BF16:
    case RSM_F16: return 2;
    case RSM_I8:
    case RSM_FP8_E4M3: return 1;
    default: return 0;
  }
}

const char* dtype_name(int dt) {
  switch (dt) {
    case RSM_F32: return "f32";
    case RSM_BF16: return "bf16";
    case RSM_F16: return "f16";
    case RSM_I8: return "i8";
    case RSM_FP8_E4M3: return "fp8_e4m3";
    default: return "?";
  }
}

struct DeviceInfo {
  bool valid = false;
  int sms = 0, smem_per_sm = 0, smem_optin = 0, smem_reserved = 0;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
constexpr size_t kNumInstances = sizeof(kInstances) / sizeof(kInstances[0]);
// largest dynamic shared memory size already configured per (device, instance),
// and the occupancy found for the last size queried (so that calls made while
// a stream is being captured issue no queries)
// (indexed by instance; then the two tensor-core variants; then the
// stochastic-rounding instances of one-byte state, at kNumInstances + 2 + instance;
// then the four one-byte tensor-core instances)
constexpr size_t kNumKernels = 2 * kNumInstances + 2 + 4;
int g_smem_set[kMaxDevices][kNumKernels];
int g_occ_smem[kMaxDevices][kNumKernels];
int g_occ_blocks[kMaxDevices][kNumKernels];

int device_info(int dev, DeviceInfo* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (dev < 0 || dev >= kMaxDevices) return fail(RSM_ECUDA, "device ordinal %d out of range", dev);
  DeviceInfo& d = g_dev[dev];
  if (!d.valid) {
    cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess) return fail(RSM_ECUDA, "device query failed: %s", cudaGetErrorString(e));
    d.valid = true;
  }
  *out = d;
  return RSM_OK;
}

bool verbose() {
  static const bool v = [] {
    const char* s = std::getenv("RSM_VERBOSE");
    return s != nullptr && s[0] != '\0' && s[0] != '0';
  }();
  return v;
}

// Whether two CTAs of `fn` (`threads` each, `smem` dynamic bytes) fit one SM by
// registers (allocated per warp in 256-register units out of 64K), shared
// memory (each CTA's static + dynamic + reserved bytes) and threads.
cudaError_t tc_two_per_sm_fit(const void* fn, int threads, int smem, const DeviceInfo& di, int* fits) {
  cudaFuncAttributes fa{};
  const cudaError_t e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  const int warps = (threads + 31) / 32;
  const int regs_per_warp = (fa.numRegs * 32 + 255) / 256 * 256;
  const bool regs_ok = 2 * warps * regs_per_warp <= 65536;
  const bool smem_ok = 2 * (static_cast<int>(fa.sharedSizeBytes) + smem + di.smem_reserved) <= di.smem_per_sm;
  const bool threads_ok = threads <= fa.maxThreadsPerBlock && 2 * threads <= 2048;
  *fits = regs_ok && smem_ok && threads_ok;
  if (verbose())
    std::fprintf(stderr, "[replayssm] two tensor-core CTAs per SM: regs %d (%s), smem %d+%zu (%s)\n", fa.numRegs,
                 regs_ok ? "fit" : "no", smem, fa.sharedSizeBytes, smem_ok ? "fit" : "no");
  return cudaSuccess;
}


// Host-side validation; returns the instance index or a negative code.
int validate(const rsm_materialize_args* a) {
  if (a == nullptr) return fail(RSM_EINVAL, "args is NULL");
  const struct {
    const void* p;
    const char* name;
  } tables[] = {
      {a->state_ptrs, "state_ptrs"},
      {a->state_slot_strides, "state_slot_strides"},
      {a->x_cache_ptrs, "x_cache_ptrs"},
      {a->x_cache_slot_strides, "x_cache_slot_strides"},
      {a->B_cache_ptrs, "B_cache_ptrs"},
      {a->B_cache_slot_strides, "B_cache_slot_strides"},
      {a->dt_cache_ptrs, "dt_cache_ptrs"},
      {a->dt_cache_slot_strides, "dt_cache_slot_strides"},
      {a->A_ptrs, "A_ptrs"},
      {a->src_slots, "src_slots"},
      {a->dst_slots, "dst_slots"},
      {a->ring_start, "ring_start"},
      {a->replay_prefix_len, "replay_prefix_len"},
      {a->active_request_indices, "active_request_indices"},
  };
  for (const auto& t : tables)
    if (t.p == nullptr) return fail(RSM_EINVAL, "%s is NULL", t.name);
  if (a->num_layers <= 0) return fail(RSM_EINVAL, "num_layers must be positive (got %d)", a->num_layers);
  if (a->batch <= 0) return fail(RSM_EINVAL, "batch must be positive (got %d)", a->batch);
  if (a->num_heads <= 0 || a->num_heads > 0x7FFFFFFFLL)
    return fail(RSM_EINVAL, "num_heads must be in [1, 2^31-1] (got %lld)", static_cast<long long>(a->num_heads));
  if (a->heads_per_group <= 0 || a->num_heads % a->heads_per_group != 0)
    return fail(RSM_EINVAL, "heads_per_group (%d) must divide num_heads (%lld)", a->heads_per_group,
                static_cast<long long>(a->num_heads));
  if (a->max_window < 1 || a->max_window > rsm::kMaxWindow)
    return fail(RSM_EINVAL, "max_window must be in [1, %d] (got %d)", rsm::kMaxWindow, a->max_window);
  if (a->ring_buffer_len < 1) return fail(RSM_EINVAL, "ring_buffer_len must be >= 1 (got %d)", a->ring_buffer_len);
  if (a->dim <= 0 || a->dstate <= 0) return fail(RSM_EINVAL, "dim and dstate must be positive");
  if (elem_bytes(a->state_dtype) == 0) return fail(RSM_EINVAL, "unknown state_dtype %d", a->state_dtype);
  if (a->input_dtype != RSM_BF16 && a->input_dtype != RSM_F32)
    return fail(RSM_EINVAL, "input_dtype must be BF16 or F32 (got %s)", dtype_name(a->input_dtype));
  if (a->matrixA_dtype != RSM_F32)
    return fail(RSM_EINVAL, "matrixA_dtype must be F32 (got %s)", dtype_name(a->matrixA_dtype));
  const bool quant = elem_bytes(a->state_dtype) == 1;
  if (quant && (a->dim != 64 || a->dstate != 128))
    return fail(RSM_EINVAL, "one-byte state requires dim=64 and dstate=128 (got %d, %d)", a->dim, a->dstate);
  if (quant && (a->state_scale_ptrs == nullptr || a->state_scale_slot_strides == nullptr))
    return fail(RSM_EINVAL, "one-byte state needs state_scale_ptrs and state_scale_slot_strides");
  if (a->philox_rounds < 0) return fail(RSM_EINVAL, "philox_rounds must be >= 0 (got %d)", a->philox_rounds);
  if (a->num_slots < 0) return fail(RSM_EINVAL, "num_slots must be >= 0 (got %d)", a->num_slots);
  if (a->philox_rounds > 0 && a->rand_seed == nullptr)
    return fail(RSM_EINVAL, "rand_seed is required when philox_rounds > 0");
  for (size_t i = 0; i < sizeof(kInstances) / sizeof(kInstances[0]); ++i) {
    const Instance& in = kInstances[i];
    if (in.sf == a->state_dtype && in.inf == a->input_dtype && in.dim == a->dim && in.dstate == a->dstate)
      return static_cast<int>(i);
  }
  return fail(RSM_ENOTSUP, "no kernel compiled for state %s, input %s, dim %d, dstate %d",
              dtype_name(a->state_dtype), dtype_name(a->input_dtype), a->dim, a->dstate);
}

// 16-bit state with bf16 inputs at 64 x 128 and windows of kTcMinWindow or
// more: the tensor-core variant (the prefix as an MMA)
bool uses_tensor_cores(const rsm_materialize_args* a) {
  return (a->state_dtype == RSM_BF16 || a->state_dtype == RSM_F16) && a->input_dtype == RSM_BF16 && a->dim == 64 &&
         a->dstate == 128 && a->max_window >= rsm::kTcMinWindow;
}

// One-byte state with bf16 inputs whose B groups hold an even number of heads:
// the one-byte tensor-core kernel (items of two heads of one group).
bool uses_q8_tensor_cores(const rsm_materialize_args* a) {
  return elem_bytes(a->state_dtype) == 1 && a->input_dtype == RSM_BF16 && a->dim == 64 && a->dstate == 128 &&
         a->heads_per_group % rsm::kQtHeads == 0;
}

struct Launch {
  const void* fn;
  int grid, threads, smem, stages;
  rsm::Params params;
};

constexpr int kSlotsPerSm = 6;      // pipeline slots per SM, over its CTAs
constexpr int kQ8SlotsPerCta = 4;   // one-byte state
// The tensor-core kernel: four per CTA where the arena holds them (prefixes up
// to 16 tokens), 2% faster than three on the 64-token ring sweep at k = 1, 4
// and 16 (measured on GB300, same box); 64-token items fill the arena at three.
constexpr int kTcSlotsPerCta = 4;
static_assert(kSlotsPerSm <= rsm::kMaxStages && kQ8SlotsPerCta <= rsm::kMaxStages && kTcSlotsPerCta <= rsm::kMaxStages,
              "slot count");

int plan_launch(const rsm_materialize_args* a, Launch* L) {
  const int inst = validate(a);
  if (inst < 0) return inst;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(RSM_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  DeviceInfo di;
  int rc = device_info(dev, &di);
  if (rc != RSM_OK) return rc;

  const bool quant = elem_bytes(a->state_dtype) == 1;
  // Items are packed into a byte arena, each taking its tile (+ scales) and
  // only its own k ring rows.  Several CTAs per SM (as many loaders in
  // flight) while each arena still holds two items of the longest window:
  // three for one-byte state (CTAs of four consumer warps), two otherwise;
  // fewer, down to one CTA with the whole shared memory, for long windows.
  const int sb = elem_bytes(a->state_dtype), ib = elem_bytes(a->input_dtype);
  const bool use_tc = uses_tensor_cores(a);
  const bool use_qt = uses_q8_tensor_cores(a);  // one-byte state on the tensor cores
  const int hpi = use_qt ? rsm::kQtHeads : 1;   // heads per work item
  const int item_min =
      static_cast<int>(rsm::item_layout(hpi * a->dim, a->dstate, sb, quant, ib, 0, true, hpi).bytes);
  const int item_max =
      static_cast<int>(rsm::item_layout(hpi * a->dim, a->dstate, sb, quant, ib, a->max_window, true, hpi).bytes);
  const bool sr_instance = quant && a->philox_rounds > 0;
  const bool q8 = quant && !use_qt;  // the four-warp one-byte kernel (both rounding modes)
  const int cw = q8 ? rsm::kQ8ConsumerWarps : rsm::kConsumerWarps;
  const int base = static_cast<int>(use_tc ? rsm::tc_arena_base(a->state_dtype)
                                    : use_qt ? rsm::qt_arena_base(a->max_window)
                                    : q8     ? rsm::kQ8ArenaBase
                                             : rsm::arena_base(a->dim, a->dstate, sb, cw));
  const int threads = use_tc ? rsm::kTcThreads : use_qt ? rsm::kQtThreads : 32 * (1 + cw);
  // (the one-byte tensor-core kernel: at most two CTAs of 256 TMEM columns per SM)
  // The tensor-core kernel places items exactly (an item follows the last one
  // where it fits), and in a B group of several heads every item after the
  // first leaves its B rows out: two consecutive items of the longest window
  // then take one item with B rows and one without.
  const int need = use_tc && a->heads_per_group > 1
                       ? item_max + static_cast<int>(rsm::item_layout(a->dim, a->dstate, sb, quant, ib, a->max_window,
                                                                      false, 1).bytes)
                       : 2 * item_max;
  int ctas = q8 ? 3 : 2, arena = 0;
  for (; ctas >= 1; --ctas) {
    const int per_cta = ctas == 1 ? di.smem_optin : di.smem_per_sm / ctas - di.smem_reserved;
    arena = (per_cta - base) / 128 * 128;
    if (arena >= need) break;
  }
  if (ctas < 1) return fail(RSM_ENOTSUP, "two work items (%d bytes) do not fit in shared memory", need);
  // Six items in flight per SM (three per CTA at two CTAs per SM): measured
  // on GB300 against two and four per CTA, it is the fastest with replay at
  // every window length (four per CTA is 2% slower on the 48-layer bf16 shape).
  // One-byte state: four per CTA (its items are half the size; two-head items
  // of the tensor-core kernel are the size of one 16-bit head).
  int stages = arena / item_min;
  const int stage_cap = q8 || use_qt ? kQ8SlotsPerCta
                        : use_tc     ? std::max(kTcSlotsPerCta, kSlotsPerSm / ctas)
                                     : kSlotsPerSm / ctas;
  if (stages > stage_cap) stages = stage_cap;
  const int smem = base + arena;
  const bool two = ctas >= 2;

  const bool fp8 = a->state_dtype == RSM_FP8_E4M3;
  const void* fn =
      use_tc   ? (a->state_dtype == RSM_BF16 ? rsm::kernel_for_tc<RSM_BF16>() : rsm::kernel_for_tc<RSM_F16>())
      : use_qt ? (fp8 ? (sr_instance ? rsm::kernel_for_q8tc<RSM_FP8_E4M3, true>()
                                     : rsm::kernel_for_q8tc<RSM_FP8_E4M3, false>())
                      : (sr_instance ? rsm::kernel_for_q8tc<RSM_I8, true>() : rsm::kernel_for_q8tc<RSM_I8, false>()))
      : sr_instance ? kInstances[inst].kernel_sr()
                    : kInstances[inst].kernel();
  const int ci = use_tc        ? static_cast<int>(kNumInstances) + (a->state_dtype == RSM_F16 ? 1 : 0)
                 : use_qt      ? static_cast<int>(2 * kNumInstances) + 2 + (fp8 ? 2 : 0) + (sr_instance ? 1 : 0)
                 : sr_instance ? static_cast<int>(kNumInstances) + 2 + inst
                               : inst;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_smem_set[dev][ci] < smem) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return fail(RSM_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      g_smem_set[dev][ci] = smem;
    }
    if (g_occ_smem[dev][ci] == smem) {
      per_sm = g_occ_blocks[dev][ci];
    } else {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
      if (e != cudaSuccess) return fail(RSM_ECUDA, "occupancy query: %s", cudaGetErrorString(e));
      if (verbose()) std::fprintf(stderr, "[replayssm] occupancy query: %d CTAs per SM\n", per_sm);
      // The occupancy query reports one CTA per SM for the tensor-core kernel,
      // while the hardware's own limits (ncu's occupancy section: shared
      // memory 2, registers 2) let two run side by side, each holding 256 of
      // the SM's 512 TMEM columns.  Two are planned only after checking those
      // limits here; were the second not co-scheduled, the persistent grid
      // would merely take a second wave.
      if ((use_tc || use_qt) && two && per_sm < 2) {
        int fits = 0;
        e = tc_two_per_sm_fit(fn, threads, smem, di, &fits);
        if (e != cudaSuccess) return fail(RSM_ECUDA, "cudaFuncGetAttributes: %s", cudaGetErrorString(e));
        if (fits) per_sm = 2;
      }
      if (use_qt && per_sm > 2) per_sm = 2;  // TMEM: 2 x 256 of 512 columns
      g_occ_smem[dev][ci] = smem;
      g_occ_blocks[dev][ci] = per_sm;
    }
  }
  if (per_sm < 1) return fail(RSM_ENOTSUP, "kernel does not fit on an SM with %d bytes of shared memory", smem);

  rsm::Params& p = L->params;
  p.state_ptrs = a->state_ptrs;
  p.state_strides = a->state_slot_strides;
  p.x_ptrs = a->x_cache_ptrs;
  p.x_strides = a->x_cache_slot_strides;
  p.B_ptrs = a->B_cache_ptrs;
  p.B_strides = a->B_cache_slot_strides;
  p.dt_ptrs = a->dt_cache_ptrs;
  p.dt_strides = a->dt_cache_slot_strides;
  p.A_ptrs = a->A_ptrs;
  p.scale_ptrs = quant ? a->state_scale_ptrs : nullptr;
  p.scale_strides = quant ? a->state_scale_slot_strides : nullptr;
  p.src_slots = a->src_slots;
  p.dst_slots = a->dst_slots;
  p.ring_start = a->ring_start;
  p.prefix_len = a->replay_prefix_len;
  p.active = a->active_request_indices;
  p.rand_seed = a->philox_rounds > 0 ? a->rand_seed : nullptr;
  p.status = a->device_status;
  p.L = a->num_layers;
  p.Bt = a->batch;
  p.H = static_cast<int32_t>(a->num_heads);
  p.hpg = a->heads_per_group;
  p.W = a->max_window;
  p.R = a->ring_buffer_len;
  p.pad = a->pad_slot_id;
  p.philox_rounds = a->philox_rounds;
  p.num_slots = a->num_slots;
  p.tc_min_k = use_tc ? rsm::kTcMinK : use_qt ? 1 : 0;
  p.desc0 = use_tc   ? rsm::tc_desc_base(a->state_dtype)
            : use_qt ? rsm::qt_desc_base(a->max_window)
            : q8     ? rsm::kQ8DescBase
                     : rsm::desc_base(a->dim, a->dstate, sb, cw);
  p.arena0 = static_cast<uint32_t>(base);
  p.arena_bytes = static_cast<uint32_t>(arena);
  p.stages = static_cast<uint32_t>(stages);

  L->fn = fn;
  L->grid = di.sms * per_sm;
  L->threads = threads;
  L->smem = smem;
  L->stages = stages;
  return RSM_OK;
}

// ---------------------------------------------------------------------------
// gated-delta-rule commit (flashinfer.gdn_decode.gated_delta_rule_replayssm_commit,
// API page: Parameters and Notes give the checks below)
// ---------------------------------------------------------------------------
int g_gdn_smem_set[kMaxDevices];
int g_gdn_occ_smem[kMaxDevices];
int g_gdn_occ_blocks[kMaxDevices];

int validate_gdn(const rsm_gdn_commit_args* a) {
  if (a == nullptr) return fail(RSM_EINVAL, "args is NULL");
  const struct {
    const void* p;
    const char* name;
  } tensors[] = {{a->checkpoint_state, "checkpoint_state"}, {a->rawv_cache, "rawv_cache"},
                 {a->rawk_cache, "rawk_cache"},             {a->g_cache, "g_cache"},
                 {a->beta_cache, "beta_cache"},             {a->state_indices, "state_indices"},
                 {a->accept_lens, "accept_lens"}};
  for (const auto& t : tensors) {
    if (t.p == nullptr) return fail(RSM_EINVAL, "%s is NULL", t.name);
    if (reinterpret_cast<uintptr_t>(t.p) % 16 != 0)
      return fail(RSM_EINVAL, "%s is not 16-byte aligned", t.name);
  }
  if ((a->track_state_indices == nullptr) != (a->track_steps == nullptr))
    return fail(RSM_EINVAL, "track_state_indices and track_steps must be given together");
  if (a->track_state_indices != nullptr &&
      (reinterpret_cast<uintptr_t>(a->track_state_indices) % 16 != 0 ||
       reinterpret_cast<uintptr_t>(a->track_steps) % 16 != 0))
    return fail(RSM_EINVAL, "track tensors are not 16-byte aligned");
  if (a->layers <= 0 || a->slots <= 0 || a->batch < 0)
    return fail(RSM_EINVAL, "layers and slots must be positive and batch non-negative");
  if (a->num_v_heads <= 0 || a->num_k_heads <= 0 || a->num_v_heads % a->num_k_heads != 0)
    return fail(RSM_EINVAL, "num_k_heads (%d) must divide num_v_heads (%d)", a->num_k_heads, a->num_v_heads);
  if (a->window < 1 || a->window > gdn::kMaxWindow)
    return fail(RSM_EINVAL, "window %d outside [1, %d]", a->window, gdn::kMaxWindow);
  if (a->null_block_id < -1) return fail(RSM_EINVAL, "null_block_id must be >= -1");
  if (a->backend < RSM_GDN_BACKEND_AUTO || a->backend > RSM_GDN_BACKEND_TCGEN05)
    return fail(RSM_EINVAL, "unknown backend %d", a->backend);
  if (a->backend == RSM_GDN_BACKEND_TCGEN05) {
    if (!a->use_qk_l2norm) return fail(RSM_EINVAL, "backend tcgen05 requires use_qk_l2norm");
    if (a->track_state_indices != nullptr) return fail(RSM_EINVAL, "backend tcgen05 does not support tracking");
    if (a->window < gdn::kTcMinT || a->window > gdn::kTcMaxT)
      return fail(RSM_EINVAL, "backend tcgen05 supports windows of %d to %d tokens (got %d)", gdn::kTcMinT,
                  gdn::kTcMaxT, a->window);
    if (static_cast<int64_t>(a->layers) * a->slots * a->num_v_heads * gdn::kDV > 0x7FFFFFFFLL)
      return fail(RSM_EINVAL, "backend tcgen05: checkpoint_state has more than 2^31 rows");
  }
  const int64_t heads = static_cast<int64_t>(a->layers) * a->slots * a->num_v_heads;
  if (heads * gdn::kDV * gdn::kDK >= (int64_t{1} << 62) / 4)
    return fail(RSM_EINVAL, "checkpoint_state is too large");
  return RSM_OK;
}

struct GdnLaunch {
  int grid, smem;
  gdn::Params params;
};

int plan_gdn(const rsm_gdn_commit_args* a, GdnLaunch* L) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(RSM_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  DeviceInfo di;
  int rc = device_info(dev, &di);
  if (rc != RSM_OK) return rc;
  // as for the materialization kernel: two CTAs per SM while each arena holds
  // two items of the longest window, six pipeline slots per SM
  const int item_min = static_cast<int>(gdn::item_layout(1).bytes);
  const int item_max = static_cast<int>(gdn::item_layout(a->window).bytes);
  const int base = static_cast<int>(gdn::kArenaOff);
  const int two_cta = di.smem_per_sm / 2 - di.smem_reserved - base;
  const int one_cta = di.smem_optin - base;
  const bool two = two_cta >= 2 * item_max;
  const int arena = (two ? two_cta : one_cta) / 128 * 128;
  if (arena < 2 * item_max) return fail(RSM_ENOTSUP, "two work items of %d bytes do not fit", item_max);
  int slots = arena / item_min;
  if (slots > kSlotsPerSm / (two ? 2 : 1)) slots = kSlotsPerSm / (two ? 2 : 1);
  const int smem = base + arena;
  const void* fn = gdn::commit_kernel();
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_gdn_smem_set[dev] < smem) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return fail(RSM_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      g_gdn_smem_set[dev] = smem;
    }
    if (g_gdn_occ_smem[dev] == smem) {
      per_sm = g_gdn_occ_blocks[dev];
    } else {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, gdn::kThreads, smem);
      if (e != cudaSuccess) return fail(RSM_ECUDA, "occupancy query: %s", cudaGetErrorString(e));
      g_gdn_occ_smem[dev] = smem;
      g_gdn_occ_blocks[dev] = per_sm;
    }
  }
  if (per_sm < 1) return fail(RSM_ENOTSUP, "kernel does not fit on an SM with %d bytes of shared memory", smem);
  gdn::Params& p = L->params;
  p.state = a->checkpoint_state;
  p.rawv = a->rawv_cache;
  p.rawk = a->rawk_cache;
  p.g = a->g_cache;
  p.beta = a->beta_cache;
  p.state_indices = a->state_indices;
  p.accept_lens = a->accept_lens;
  p.track_indices = a->track_state_indices;
  p.track_steps = a->track_steps;
  p.status = a->device_status;
  p.L = a->layers;
  p.SL = a->slots;
  p.HV = a->num_v_heads;
  p.H = a->num_k_heads;
  p.T = a->window;
  p.B = a->batch;
  p.l2norm = a->use_qk_l2norm != 0;
  p.null_id = a->null_block_id;
  p.arena_bytes = static_cast<uint32_t>(arena);
  p.slots = static_cast<uint32_t>(slots);
  L->grid = di.sms * per_sm;
  L->smem = smem;
  return RSM_OK;
}

// The tcgen05 backend: one CTA per SM with the opt-in shared memory, and a
// tensor map over checkpoint_state viewed as [layers*slots*HV*128 rows, 128]
// fp32 (boxes of 128 rows x 32 columns, 128-byte swizzle), encoded per call
// through the driver's entry point (no link against the driver library).
using TensorMapEncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                       const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                       CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

TensorMapEncodeFn tensor_map_encoder() {
  static const TensorMapEncodeFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<TensorMapEncodeFn>(nullptr);
    return reinterpret_cast<TensorMapEncodeFn>(f);
  }();
  return fn;
}

int g_gdn_tc_smem_set[kMaxDevices];

int launch_gdn_tc(const rsm_gdn_commit_args* a, void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(RSM_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  DeviceInfo di;
  int rc = device_info(dev, &di);
  if (rc != RSM_OK) return rc;
  const int item_min = static_cast<int>(gdn::tc_item_layout(1).bytes);
  const int item_max = static_cast<int>(gdn::tc_item_layout(a->window).bytes);
  const int arena = (di.smem_optin - static_cast<int>(gdn::kTcArenaOff)) / 1024 * 1024;
  if (arena < 2 * item_max) return fail(RSM_ENOTSUP, "two work items of %d bytes do not fit", item_max);
  int slots = arena / item_min;
  if (slots > 4) slots = 4;
  const int smem = static_cast<int>(gdn::kTcArenaOff) + arena;
  const TensorMapEncodeFn encode = tensor_map_encoder();
  if (encode == nullptr) return fail(RSM_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");

  gdn::TcParams tp{};
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(gdn::kDK),
                              static_cast<cuuint64_t>(a->layers) * a->slots * a->num_v_heads * gdn::kDV};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(gdn::kDK) * 4u};
  const cuuint32_t box[2] = {32u, static_cast<cuuint32_t>(gdn::kDV)};
  const cuuint32_t elem_strides[2] = {1u, 1u};
  const CUresult cr = encode(&tp.tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2u, a->checkpoint_state, dims, strides, box,
                             elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return fail(RSM_ECUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(cr));

  gdn::Params& p = tp.p;
  p.state = a->checkpoint_state;
  p.rawv = a->rawv_cache;
  p.rawk = a->rawk_cache;
  p.g = a->g_cache;
  p.beta = a->beta_cache;
  p.state_indices = a->state_indices;
  p.accept_lens = a->accept_lens;
  p.track_indices = nullptr;
  p.track_steps = nullptr;
  p.status = a->device_status;
  p.L = a->layers;
  p.SL = a->slots;
  p.HV = a->num_v_heads;
  p.H = a->num_k_heads;
  p.T = a->window;
  p.B = a->batch;
  p.l2norm = 1;
  p.null_id = a->null_block_id;
  p.arena_bytes = static_cast<uint32_t>(arena);
  p.slots = static_cast<uint32_t>(slots);

  const void* fn = gdn::commit_tc_kernel();
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_gdn_tc_smem_set[dev] < smem) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return fail(RSM_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      g_gdn_tc_smem_set[dev] = smem;
    }
  }
  if (verbose())
    std::fprintf(stderr, "[replayssm] gdn commit (tcgen05) grid=%d block=%d smem=%d slots=%d\n", di.sms,
                 gdn::kTcThreads, smem, slots);
  void* kargs[] = {&tp};
  e = cudaLaunchKernel(fn, dim3(di.sms), dim3(gdn::kTcThreads), kargs, static_cast<size_t>(smem),
                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(RSM_ECUDA, "launch failed: %s", cudaGetErrorString(e));
  g_last_error.clear();
  return RSM_OK;
}

}  // namespace

extern "C" {

int rsm_materialize(const rsm_materialize_args* args, void* stream) {
  Launch L;
  const int rc = plan_launch(args, &L);
  if (rc != RSM_OK) return rc;
  if (verbose())
    std::fprintf(stderr, "[replayssm] state=%s input=%s dim=%d dstate=%d grid=%d block=%d smem=%d stages=%d\n",
                 dtype_name(args->state_dtype), dtype_name(args->input_dtype), args->dim, args->dstate, L.grid,
                 L.threads, L.smem, L.stages);
  void* kargs[] = {&L.params};
  cudaError_t e = cudaLaunchKernel(L.fn, dim3(L.grid), dim3(L.threads), kargs, static_cast<size_t>(L.smem),
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(RSM_ECUDA, "launch failed: %s", cudaGetErrorString(e));
  g_last_error.clear();
  return RSM_OK;
}

int rsm_launch_config(const rsm_materialize_args* args, int* grid, int* block, int* smem_bytes, int* stages) {
  Launch L;
  const int rc = plan_launch(args, &L);
  if (rc != RSM_OK) return rc;
  if (grid) *grid = L.grid;
  if (block) *block = L.threads;
  if (smem_bytes) *smem_bytes = L.smem;
  if (stages) *stages = L.stages;
  return RSM_OK;
}

int rsm_gdn_commit(const rsm_gdn_commit_args* args, void* stream) {
  int rc = validate_gdn(args);
  if (rc != RSM_OK) return rc;
  if (args->batch == 0) {
    g_last_error.clear();
    return RSM_OK;
  }
  if (args->backend == RSM_GDN_BACKEND_TCGEN05) return launch_gdn_tc(args, stream);
  GdnLaunch L;
  rc = plan_gdn(args, &L);
  if (rc != RSM_OK) return rc;
  if (verbose())
    std::fprintf(stderr, "[replayssm] gdn commit grid=%d block=%d smem=%d slots=%u\n", L.grid, gdn::kThreads, L.smem,
                 L.params.slots);
  void* kargs[] = {&L.params};
  cudaError_t e = cudaLaunchKernel(gdn::commit_kernel(), dim3(L.grid), dim3(gdn::kThreads), kargs,
                                   static_cast<size_t>(L.smem), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(RSM_ECUDA, "launch failed: %s", cudaGetErrorString(e));
  g_last_error.clear();
  return RSM_OK;
}

const char* rsm_kernel_name(const rsm_materialize_args* args) {
  if (validate(args) < 0) return "";
  if (uses_tensor_cores(args)) return "materialize_tc_kernel";
  if (uses_q8_tensor_cores(args)) return "materialize_q8tc_kernel";
  return elem_bytes(args->state_dtype) == 1 ? "materialize_q8_kernel" : "materialize_kernel";
}

int rsm_gdn_args_size(void) { return static_cast<int>(sizeof(rsm_gdn_commit_args)); }

const char* rsm_last_error(void) { return g_last_error.c_str(); }

int rsm_args_size(void) { return static_cast<int>(sizeof(rsm_materialize_args)); }

int rsm_abi_version(void) { return RSM_ABI_VERSION; }

}  // extern "C"
