// C entry points declared in include/pkv.h: argument validation, workspace carving,
// the per-device error word, dispatch to the kernel launchers.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace pkv {

// Or-ed PKV_DEVERR_* bits, one word per device (module-scope device variable).
static __device__ unsigned int g_error_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxDecodeCtas = 1 << 16;  // largest decode grid a call may ask for
std::once_flag g_dev_once[kMaxDevices];
unsigned int* g_err_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];
std::atomic<int> g_decode_ctas_override{0};
std::atomic<int> g_decode_kernel{0};
std::atomic<int> g_prefill_kernel{0};
std::atomic<int> g_overlap{1};
std::atomic<int> g_fault{0};
SideStream g_side[kMaxDevices];
std::mutex g_side_lock[kMaxDevices];
constexpr int kNumKernels = 5;
std::atomic<void*> g_events[kNumKernels][2];

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

// Once per device, with that device current: the device address of the error word and
// the SM count.
bool device_setup(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return false;
  std::call_once(g_dev_once[dev], [dev]() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess) g_err_ptr[dev] = static_cast<unsigned int*>(p);
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) g_sm_count[dev] = n;
    // the second stream for prefill tiles beside the decode, and its fork/join events
    SideStream& sd = g_side[dev];
    if (cudaStreamCreateWithFlags(&sd.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      sd.stream = nullptr;
    }
    sd.lock = &g_side_lock[dev];
  });
  return g_err_ptr[dev] != nullptr && g_sm_count[dev] > 0;
}

// A RoPE base whose frequency table builds: finite, positive, and not so small that the
// largest frequency (below 1 / theta for theta < 1) times 2^64 / (2 pi) overflows a double.
bool rope_theta_ok(double theta) {
  return theta > 0.0 && std::isfinite(theta) && (theta >= 1.0 || std::isfinite(2.9358905032820014e+18 / theta));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Rows (t, h) of length d at offsets t*st + h*sh never overlap: token-major or head-major.
bool rows_disjoint(int64_t T, int64_t st, int64_t H, int64_t sh, int64_t d) {
  if (T <= 1 && H <= 1) return true;
  if (H <= 1) return st >= d;
  if (T <= 1) return sh >= d;
  return (sh >= d && st >= (H - 1) * sh + d) || (st >= d && sh >= (T - 1) * st + d);
}

}  // namespace

int device_sm_count() {
  const int dev = current_device();
  return device_setup(dev) ? g_sm_count[dev] : 0;
}

void record_kernel_event(int which, bool after, cudaStream_t stream) {
  if (which <= 0 || which >= kNumKernels) return;
  void* e = g_events[which][after ? 1 : 0].load();
  if (e) cudaEventRecord(static_cast<cudaEvent_t>(e), stream);
}

int decode_kernel_choice() { return g_decode_kernel.load(); }

int overlap_choice() { return g_overlap.load(); }

int fault_injection_choice() { return g_fault.load(); }

bool side_stream_for_device(SideStream* s) {
  const int dev = current_device();
  if (!device_setup(dev) || g_side[dev].stream == nullptr) return false;
  *s = g_side[dev];
  return true;
}

// Automatic choice: the tcgen05 tiles (33 us vs 113 us for the mma.sync tiles on the
// mixed chunked-prefill workload on GB300, both on all SMs).
int prefill_kernel_choice() {
  const int k = g_prefill_kernel.load();
  return k == 0 ? 2 : k;
}

int decode_ctas_for_device() {
  const int o = g_decode_ctas_override.load();
  if (o > 0) return o;
  return device_sm_count();
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL: return "a required pointer is NULL";
    case PKV_ERR_SHAPE: return "invalid or inconsistent sizes";
    case PKV_ERR_STRIDE: return "unsupported stride";
    case PKV_ERR_ALIGN: return "pointer or stride breaks 16-byte row alignment";
    case PKV_ERR_UNSUPPORTED: return "head_dim / block_size / head counts outside the compiled set";
    case PKV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

int pkv_version(void) { return 200; }

int pkv_set_overlap(int on) {
  if (on != 0 && on != 1) return PKV_ERR_SHAPE;
  g_overlap.store(on);
  return PKV_OK;
}

int pkv_set_fault_injection(int kind) {
  if (kind != 0 && kind != PKV_FAULT_DECODE_NO_COPIES && kind != PKV_FAULT_PLAN_NO_READY) return PKV_ERR_SHAPE;
  g_fault.store(kind);
  return PKV_OK;
}

int pkv_set_decode_ctas(int32_t ctas) {
  if (ctas < 0 || ctas > kMaxDecodeCtas) return PKV_ERR_SHAPE;
  g_decode_ctas_override.store(ctas);
  return PKV_OK;
}

int pkv_set_decode_kernel(int kind) {
  if (kind < 0 || kind > 2) return PKV_ERR_SHAPE;
  g_decode_kernel.store(kind);
  return PKV_OK;
}

int pkv_set_prefill_kernel(int kind) {
  if (kind < 0 || kind > 2) return PKV_ERR_SHAPE;
  g_prefill_kernel.store(kind);
  return PKV_OK;
}

int pkv_set_kernel_events(int which, void* start_event, void* stop_event) {
  if (which < 0 || which >= kNumKernels) return PKV_ERR_SHAPE;
  if (which == 0) {
    for (int k = 1; k < kNumKernels; ++k) g_events[k][0] = g_events[k][1] = nullptr;
    return PKV_OK;
  }
  const bool on = start_event && stop_event;
  g_events[which][0] = on ? start_event : nullptr;
  g_events[which][1] = on ? stop_event : nullptr;
  return PKV_OK;
}

int pkv_kv_append(void* q, int64_t q_st, int64_t q_sh, const void* k, int64_t k_st, int64_t k_sh,
                  const void* v, int64_t v_st, int64_t v_sh, const int64_t* positions,
                  const int64_t* slot_mapping, void* k_cache, void* v_cache, int64_t num_tokens,
                  int64_t num_q_heads, int64_t num_kv_heads, int64_t head_dim, int64_t num_blocks,
                  int64_t block_size, double rope_theta, void* stream) {
  if (num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks < 0) return PKV_ERR_SHAPE;
  if (num_q_heads % num_kv_heads) return PKV_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  const int bs_log2 = block_size_log2(block_size);
  if (bs_log2 < 0) return PKV_ERR_UNSUPPORTED;
  if (num_blocks > INT32_MAX) return PKV_ERR_SHAPE;  // block ids are int32
  if (!rope_theta_ok(rope_theta)) return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!q || !k || !v || !positions || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_NULL;
  if (q_st < 0 || q_sh < 0 || k_st < 0 || k_sh < 0 || v_st < 0 || v_sh < 0) return PKV_ERR_STRIDE;
  if (!rows_disjoint(num_tokens, q_st, num_q_heads, q_sh, head_dim)) return PKV_ERR_STRIDE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_ALIGN;
  if ((q_st | q_sh | k_st | k_sh | v_st | v_sh) & 7) return PKV_ERR_ALIGN;
  const int dev = current_device();
  if (!device_setup(dev)) return PKV_ERR_CUDA;
  AppendArgs a{};
  a.q = q;
  a.q_st = q_st;
  a.q_sh = q_sh;
  a.k = k;
  a.k_st = k_st;
  a.k_sh = k_sh;
  a.v = v;
  a.v_st = v_st;
  a.v_sh = v_sh;
  a.positions = positions;
  a.slots = slot_mapping;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.num_tokens = num_tokens;
  a.num_slots = num_blocks << bs_log2;
  a.bs_log2 = bs_log2;
  a.hq = static_cast<int>(num_q_heads);
  a.hkv = static_cast<int>(num_kv_heads);
  a.head_dim = static_cast<int>(head_dim);
  a.theta = rope_theta;
  a.err = g_err_ptr[dev];
  return launch_kv_append(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int pkv_kv_append_paged(void* q, int64_t q_st, int64_t q_sh, const void* k, int64_t k_st, int64_t k_sh,
                        const void* v, int64_t v_st, int64_t v_sh, const int32_t* block_tables, int64_t bt_stride,
                        int64_t max_blocks_per_seq, const int32_t* context_lens, const int32_t* query_start_loc,
                        int64_t num_seqs, void* k_cache, void* v_cache, int64_t num_tokens, int64_t num_q_heads,
                        int64_t num_kv_heads, int64_t head_dim, int64_t num_blocks, int64_t block_size,
                        double rope_theta, int64_t* positions_out, int64_t* slot_mapping_out, void* stream) {
  if (num_tokens < 0 || num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks < 0 ||
      max_blocks_per_seq < 0)
    return PKV_ERR_SHAPE;
  if (num_q_heads % num_kv_heads) return PKV_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  const int bs_log2 = block_size_log2(block_size);
  if (bs_log2 < 0) return PKV_ERR_UNSUPPORTED;
  if (num_blocks > INT32_MAX) return PKV_ERR_SHAPE;  // block ids are int32
  if (!rope_theta_ok(rope_theta)) return PKV_ERR_SHAPE;
  if (num_seqs > (1 << 30)) return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!q || !k || !v || !block_tables || !context_lens || !query_start_loc || !k_cache || !v_cache)
    return PKV_ERR_NULL;
  if (bt_stride < max_blocks_per_seq) return PKV_ERR_STRIDE;
  if (q_st < 0 || q_sh < 0 || k_st < 0 || k_sh < 0 || v_st < 0 || v_sh < 0) return PKV_ERR_STRIDE;
  if (!rows_disjoint(num_tokens, q_st, num_q_heads, q_sh, head_dim)) return PKV_ERR_STRIDE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_ALIGN;
  if ((q_st | q_sh | k_st | k_sh | v_st | v_sh) & 7) return PKV_ERR_ALIGN;
  const int dev = current_device();
  if (!device_setup(dev)) return PKV_ERR_CUDA;
  AppendArgs a{};
  a.q = q;
  a.q_st = q_st;
  a.q_sh = q_sh;
  a.k = k;
  a.k_st = k_st;
  a.k_sh = k_sh;
  a.v = v;
  a.v_st = v_st;
  a.v_sh = v_sh;
  a.qsl = query_start_loc;
  a.context_lens = context_lens;
  a.block_tables = block_tables;
  a.bt_stride = bt_stride;
  a.max_blocks = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.positions_out = positions_out;
  a.slots_out = slot_mapping_out;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.num_tokens = num_tokens;
  a.num_slots = num_blocks << bs_log2;
  a.bs_log2 = bs_log2;
  a.hq = static_cast<int>(num_q_heads);
  a.hkv = static_cast<int>(num_kv_heads);
  a.head_dim = static_cast<int>(head_dim);
  a.theta = rope_theta;
  a.err = g_err_ptr[dev];
  return launch_kv_append(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int pkv_rope_turn_table(double rope_theta, int64_t head_dim, uint64_t* out) {
  if (!out) return PKV_ERR_NULL;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  unsigned long long F[kMaxHeadDim / 2];
  if (!rope_turn_table(rope_theta, static_cast<int>(head_dim), F)) return PKV_ERR_SHAPE;
  for (int64_t i = 0; i < head_dim / 2; ++i) out[i] = F[i];
  return PKV_OK;
}

size_t pkv_paged_attention_workspace_size_ex(int64_t num_tokens, int64_t num_seqs, int64_t num_q_heads,
                                             int64_t num_kv_heads, int64_t head_dim, int64_t max_blocks_per_seq,
                                             int32_t decode_ctas) {
  if (num_tokens < 0 || num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq < 0)
    return 0;
  if (head_dim != 64 && head_dim != 128) return 0;
  if (decode_ctas < 0 || decode_ctas > kMaxDecodeCtas) return 0;
  const int ctas = decode_ctas > 0 ? decode_ctas : decode_ctas_for_device();
  if (ctas <= 0) return 0;
  return plan_sizes(num_tokens, num_seqs, num_q_heads, head_dim, ctas).total;
}

size_t pkv_paged_attention_workspace_size(int64_t num_tokens, int64_t num_seqs, int64_t num_q_heads,
                                          int64_t num_kv_heads, int64_t head_dim,
                                          int64_t max_blocks_per_seq) {
  return pkv_paged_attention_workspace_size_ex(num_tokens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                               max_blocks_per_seq, 0);
}

}  // extern "C"

namespace {

int paged_attention_impl(const void* q, int64_t q_st, int64_t q_sh, const void* k_cache, const void* v_cache,
                         int64_t num_blocks, int64_t block_size, const int32_t* block_tables, int64_t bt_stride,
                         int64_t max_blocks_per_seq, const int32_t* context_lens, const int32_t* query_start_loc,
                         int64_t num_seqs, void* out, int64_t o_st, int64_t o_sh, int64_t num_tokens,
                         int64_t num_q_heads, int64_t num_kv_heads, int64_t head_dim, float scale, void* workspace,
                         size_t workspace_bytes, void* stream, const pkv_attention_options* opt) {
  if (opt) {
    if (opt->struct_size != sizeof(pkv_attention_options)) return PKV_ERR_SHAPE;
    if (opt->decode_kernel < 0 || opt->decode_kernel > 2 || opt->prefill_kernel < 0 || opt->prefill_kernel > 2 ||
        opt->overlap < 0 || opt->overlap > 2 || opt->decode_ctas < 0 || opt->decode_ctas > kMaxDecodeCtas ||
        (opt->flags & ~(PKV_ATTN_PLAN_EARLY | PKV_ATTN_STREAM_EARLY)) != 0)
      return PKV_ERR_SHAPE;
    const int given = (opt->side_stream != nullptr) + (opt->fork_event != nullptr) + (opt->join_event != nullptr);
    if (given != 0 && given != 3) return PKV_ERR_NULL;
  }
  if (num_tokens < 0 || num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks < 0 ||
      max_blocks_per_seq < 0)
    return PKV_ERR_SHAPE;
  if (num_q_heads % num_kv_heads) return PKV_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  const int bs_log2 = block_size_log2(block_size);
  if (bs_log2 < 0) return PKV_ERR_UNSUPPORTED;
  if (num_blocks > INT32_MAX) return PKV_ERR_SHAPE;  // block ids are int32
  if (kDecodeWarps % num_kv_heads) return PKV_ERR_UNSUPPORTED;
  const int64_t group = num_q_heads / num_kv_heads;
  if (group < 1 || group > 8) return PKV_ERR_UNSUPPORTED;
  if (num_seqs > (1 << 24) || num_tokens > (1 << 28) || max_blocks_per_seq > (1 << 24)) return PKV_ERR_SHAPE;
  if (num_tokens == 0 || num_seqs == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start_loc || !out)
    return PKV_ERR_NULL;
  if (bt_stride < max_blocks_per_seq) return PKV_ERR_STRIDE;
  if (q_st < 0 || q_sh < 0 || o_st < 0 || o_sh < 0) return PKV_ERR_STRIDE;
  if (!rows_disjoint(num_tokens, o_st, num_q_heads, o_sh, head_dim)) return PKV_ERR_STRIDE;
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ALIGN;
  if ((q_st | q_sh | o_st | o_sh) & 7) return PKV_ERR_ALIGN;
  const int dev = current_device();
  if (!device_setup(dev)) return PKV_ERR_CUDA;
  const int ctas = (opt && opt->decode_ctas > 0) ? opt->decode_ctas : decode_ctas_for_device();
  const PlanSizes ps = plan_sizes(num_tokens, num_seqs, num_q_heads, head_dim, ctas);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < ps.total)
    return PKV_ERR_WORKSPACE;
  AttnArgs a;
  a.q = q;
  a.q_st = q_st;
  a.q_sh = q_sh;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.num_blocks = num_blocks;
  a.bs_log2 = bs_log2;
  a.block_tables = block_tables;
  a.bt_stride = bt_stride;
  a.max_blocks = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.qsl = query_start_loc;
  a.num_seqs = num_seqs;
  a.out = out;
  a.o_st = o_st;
  a.o_sh = o_sh;
  a.num_tokens = num_tokens;
  a.hq = static_cast<int>(num_q_heads);
  a.hkv = static_cast<int>(num_kv_heads);
  a.head_dim = static_cast<int>(head_dim);
  a.scale = scale;
  a.decode_ctas = ctas;
  a.decode_kernel = (opt && opt->decode_kernel) ? opt->decode_kernel : decode_kernel_choice();
  a.prefill_kernel = (opt && opt->prefill_kernel) ? opt->prefill_kernel : prefill_kernel_choice();
  a.overlap = (opt && opt->overlap) ? (opt->overlap == 1 ? 1 : 0) : overlap_choice();
  a.fault = fault_injection_choice();
  const int flags = opt ? opt->flags : 0;
  // early streaming needs the one-CTA planner (up to kSmallPlanMaxSeqs sequences), which
  // publishes the plan; it implies early planning
  a.stream_early = (flags & PKV_ATTN_STREAM_EARLY) && num_seqs <= kSmallPlanMaxSeqs ? 1 : 0;
  a.plan_early = (flags & (PKV_ATTN_PLAN_EARLY | PKV_ATTN_STREAM_EARLY)) ? 1 : 0;
  a.side_stream = opt ? static_cast<cudaStream_t>(opt->side_stream) : nullptr;
  a.fork_event = opt ? static_cast<cudaEvent_t>(opt->fork_event) : nullptr;
  a.join_event = opt ? static_cast<cudaEvent_t>(opt->join_event) : nullptr;
  a.plan = plan_view(workspace, ps);
  a.max_tiles = ps.max_tiles;
  a.err = g_err_ptr[dev];
  return launch_paged_attention(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

extern "C" {

int pkv_paged_attention(const void* q, int64_t q_st, int64_t q_sh, const void* k_cache,
                        const void* v_cache, int64_t num_blocks, int64_t block_size,
                        const int32_t* block_tables, int64_t bt_stride, int64_t max_blocks_per_seq,
                        const int32_t* context_lens, const int32_t* query_start_loc, int64_t num_seqs,
                        void* out, int64_t o_st, int64_t o_sh, int64_t num_tokens, int64_t num_q_heads,
                        int64_t num_kv_heads, int64_t head_dim, float scale, void* workspace,
                        size_t workspace_bytes, void* stream) {
  return paged_attention_impl(q, q_st, q_sh, k_cache, v_cache, num_blocks, block_size, block_tables, bt_stride,
                              max_blocks_per_seq, context_lens, query_start_loc, num_seqs, out, o_st, o_sh,
                              num_tokens, num_q_heads, num_kv_heads, head_dim, scale, workspace, workspace_bytes,
                              stream, nullptr);
}

int pkv_paged_attention_ex(const void* q, int64_t q_st, int64_t q_sh, const void* k_cache,
                           const void* v_cache, int64_t num_blocks, int64_t block_size,
                           const int32_t* block_tables, int64_t bt_stride, int64_t max_blocks_per_seq,
                           const int32_t* context_lens, const int32_t* query_start_loc, int64_t num_seqs,
                           void* out, int64_t o_st, int64_t o_sh, int64_t num_tokens, int64_t num_q_heads,
                           int64_t num_kv_heads, int64_t head_dim, float scale, void* workspace,
                           size_t workspace_bytes, void* stream, const pkv_attention_options* options) {
  return paged_attention_impl(q, q_st, q_sh, k_cache, v_cache, num_blocks, block_size, block_tables, bt_stride,
                              max_blocks_per_seq, context_lens, query_start_loc, num_seqs, out, o_st, o_sh,
                              num_tokens, num_q_heads, num_kv_heads, head_dim, scale, workspace, workspace_bytes,
                              stream, options);
}

int pkv_get_device_error(uint32_t* bits, int clear, void* stream) {
  if (!bits) return PKV_ERR_NULL;
  const int dev = current_device();
  if (!device_setup(dev)) return PKV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int host = 0;
  if (cudaMemcpyAsync(&host, g_err_ptr[dev], sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
  *bits = host;
  if (clear) {
    if (cudaMemsetAsync(g_err_ptr[dev], 0, sizeof(unsigned int), s) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // extern "C"
