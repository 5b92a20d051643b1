// Internal interface between the C entry points (abi.cu) and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

namespace pkv {

// The kernels walk a sequence's keys in pages of 16 tokens whatever the pool's block size:
// the pool's blocks hold 2^k tokens, 8 <= 2^k <= 128, so a page is a 16-row piece of one
// block (block_size >= 16) or two whole blocks (block_size 8).
constexpr int kPageTokens = 16;
constexpr int kMinBlockSize = 8;
constexpr int kMaxBlockSize = 128;
// log2(block_size) for a supported block size, else -1.
inline int block_size_log2(int64_t bs) {
  for (int l = 3; (1 << l) <= kMaxBlockSize; ++l)
    if (bs == (int64_t(1) << l)) return l;
  return -1;
}
constexpr int kDecodeWarps = 8;      // consumer warps of the decode split-K kernel
constexpr int kPrefillTileQ = 64;    // query rows per mma.sync prefill work tile
constexpr int kTcPrefillRows = 128;  // rows of a tcgen05 prefill tile: floor(128 / G) positions x G heads
constexpr int kMinPrefillTileQ = kTcPrefillRows / 8;  // fewest positions per tile (G = 8): sizes the tile list
constexpr int kMaxHeadDim = 128;
// GQA group size from which the decode runs on the tensor cores by default.  Measured on
// GB300: the tensor-core variant is at least as fast for every group size (0.87 vs 0.80 of
// HBM peak at G = 2, 0.89 vs 0.21 at G = 7), so it is the default for all of them.
constexpr int kTensorDecodeMinGroup = 1;

// ---------------------------------------------------------------- work plan layout
// The planner kernel fills these arrays in the caller's workspace; the decode, prefill
// and merge kernels read them.  All offsets are 256-byte aligned.
//
// header[0] number of decode entries (spans of one row; with no prefill kernel, also one entry
//           per row of a longer span)                           n_dec
// header[1] total decode work units                            U
// header[2] work units per decode CTA                          W = ceil(U / C)
// header[3] number of prefill (seq, q-tile) work items         n_tiles
// header[4] partial-result slots in use                        S
// header[5] prefill CTAs that take work items                  P (the rest leave at once)
// header[8] plan ready word (kPlanReadyWord), written only when the decode streams early:
//           0 while the plan is being written, then 1 (new keys only in each decode entry's
//           last 16-token page) or 2 (some entry has new keys before its last page)
//
// A decode work unit is one page group of one sequence: P = kDecodeWarps / Hkv
// consecutive 16-token pages (kPageTokens), all kv heads.  Decode CTA c owns units [c W, (c+1) W) of
// the concatenation of all decode sequences' units.
constexpr int kPlanReadyWord = 8;
constexpr int kSmallPlanMaxSeqs = 1024;
constexpr long long kPlanReadySpinClocks = 1ll << 24;  // a decode CTA's wait for the ready word  // batches the one-CTA, one-thread-per-sequence planner takes
struct Plan {
  int* header;      // [16]
  int* dec_seq;     // [B]      decode list: sequence id
  int* dec_unit;    // [B + 1]  exclusive prefix of work units over the decode list
  int* dec_slot;    // [B]      first partial slot of each decode sequence
  int* dec_chunks;  // [B]      number of decode CTAs that touch the sequence
  int* dec_count;   // [B]      split states written so far (zeroed by the planner)
  int* dec_ctx;     // [B]      keys the entry's query row sees (its context, or for a prefill
                    //          row computed by the decode path, ctx - n + r + 1)
  int* dec_tq;      // [B]      the entry's query row (token index)
  int4* cta_rec;    // [C][2]   decode CTA c's start record: {entry i holding its first unit c W,
                    //          dec_unit[i], dec_unit[i + 1], sequence}, {context, query row, 0, 0}
                    //          (written only for CTAs that have units)
  int* pf_seq;      // [max_tiles]  prefill work item: sequence id
  int* pf_tile;     // [max_tiles]  prefill work item: q-tile index within the span
  float* part_ml;   // [S_max][Hq][2]   split state: running max (log2 domain), sum of weights
  float* part_acc;  // [S_max][Hq][D]   split state: unnormalised weighted sum of V
};

struct PlanSizes {
  int64_t num_seqs, num_tokens, num_q_heads, head_dim, decode_ctas;
  int64_t max_tiles, max_slots;
  size_t off_header, off_dec_seq, off_dec_unit, off_dec_slot, off_dec_chunks, off_dec_count, off_dec_ctx,
      off_dec_tq, off_cta_rec;
  size_t off_pf_seq, off_pf_tile, off_part_ml, off_part_acc, total;
};

PlanSizes plan_sizes(int64_t num_tokens, int64_t num_seqs, int64_t num_q_heads, int64_t head_dim,
                     int64_t decode_ctas);
Plan plan_view(void* workspace, const PlanSizes& s);

// ------------------------------------------------------------------------ launchers
struct AppendArgs {
  void* q;
  int64_t q_st, q_sh;
  const void* k;
  int64_t k_st, k_sh;
  const void* v;
  int64_t v_st, v_sh;
  const int64_t* positions;  // explicit positions / slots, or
  const int64_t* slots;
  const int32_t* qsl;           // (non-null) derive them from the scheduler's tables
  const int32_t* context_lens;
  const int32_t* block_tables;
  int64_t bt_stride, max_blocks, num_seqs;
  int64_t* positions_out;       // optional copies of the derived values
  int64_t* slots_out;
  void* k_cache;
  void* v_cache;
  int64_t num_tokens, num_slots;
  int bs_log2;  // log2 of the pool's block size
  int hq, hkv, head_dim;
  double theta;
  unsigned int* err;
};
cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t stream);
// The kv_append rotation frequencies as 0.64 fixed-point turn fractions F[0 .. head_dim/2);
// false for a theta that is not finite and positive, whose table does not build, or a head_dim
// outside {64, 128}.
bool rope_turn_table(double theta, int head_dim, unsigned long long* F);

struct AttnArgs {
  const void* q;
  int64_t q_st, q_sh;
  const void* k_cache;
  const void* v_cache;
  int64_t num_blocks;
  int bs_log2;  // log2 of the pool's block size
  const int32_t* block_tables;
  int64_t bt_stride, max_blocks;
  const int32_t* context_lens;
  const int32_t* qsl;
  int64_t num_seqs;
  void* out;
  int64_t o_st, o_sh;
  int64_t num_tokens;
  int hq, hkv, head_dim;
  float scale;
  int decode_ctas;
  int decode_kernel;   // 0 automatic, 1 CUDA-core (warp-shuffle), 2 tensor-core (mma.sync)
  int prefill_kernel;  // 1 mma.sync tiles, 2 tcgen05 tiles (resolved from the process setting)
  int overlap;         // 1: prefill tiles run beside the decode on a second stream (SMs split)
  int fault;           // test-only fault injection (pkv_set_fault_injection); 0 in normal use
  int plan_early;      // 1: the planner computes before waiting on the previous kernel (PKV_ATTN_PLAN_EARLY)
  int stream_early;    // 1: the plan is published at once and the tensor-core decode streams the
                       // pages without new keys before the previous kernel ends (PKV_ATTN_STREAM_EARLY)
  cudaStream_t side_stream;  // the caller's second stream for the prefill beside the decode, or null
  cudaEvent_t fork_event, join_event;  // (with it) the caller's events ordering that stream
  Plan plan;
  int64_t max_tiles;
  unsigned int* err;
};
cudaError_t launch_paged_attention(const AttnArgs& a, cudaStream_t stream);
// The tensor-core decode for each pool block size (decode_tc.cu, built once per size).
cudaError_t launch_decode_tc_bs8(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_decode_tc_bs16(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_decode_tc_bs32(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_decode_tc_bs64(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_decode_tc_bs128(const AttnArgs& a, cudaStream_t stream);

int device_sm_count();

// ------------------------------------------------------ prefill beside the decode
// A batch with prefill spans runs its prefill tiles on a second stream while the decode
// runs, each kernel on its own share of the SMs: the decode is bound by HBM and reaches
// its rate on about 120 of GB300's 152 SMs (measured: 153.9 us at 112 CTAs, 153.6 us at 152
// on the 256-sequence batch), while the prefill tiles are bound by what each SM can take
// in (TMA boxes of one kv head's rows).  The planner picks the prefill share P that
// minimises max(decode time on C - P SMs, prefill time on P SMs) with this model:
//   decode:  U units x unit bytes / min(HBM rate, SMs x per-SM decode rate)
//   prefill: max(key tiles / P, largest item's key tiles) x tile bytes / per-SM prefill rate
// Rates in bytes per ns (= GB/s), measured on GB300.  The split only moves work between
// SMs: every CTA computes what it would compute in the serial order.
constexpr float kSplitHbmBytesPerNs = 6500.f;
constexpr float kSplitDecodeSmBytesPerNs = 58.f;
// The prefill tiles' pace per SM, measured beside the decode on GB300 (mixed chunked-prefill
// batch): about 1.95 us per 128-key K/V tile of 64 KB, i.e. 33.5 GB/s per SM, at 16-, 32-, 64-
// and 128-token blocks alike (the tile's TMA boxes grow with the block, the pace does not),
// and 29 GB/s at 8-token blocks (two half-height boxes per page).  Since items follow one
// another without a CTA barrier the kernel runs about 1.14x faster there, but the split keeps
// these rates: the decode gains nothing from the SMs a higher rate would move to it, while the
// prefill then ends later than the decode (mixed step on GB300: 147.6 us at 33.5, 149.9 at 38,
// 158.6 at 42 GB/s per SM).
inline float split_prefill_sm_bytes_per_ns(int bs_log2) { return bs_log2 <= 3 ? 29.f : 33.5f; }

struct SplitArgs {
  int on;             // 1: the planner splits `sms` CTAs between prefill and decode
  int sms;            // CTAs to share out (one per SM)
  int pf_grid;        // CTAs the prefill kernel is launched with
  int hkv;            // prefill items per q tile (one per kv head)
  float unit_bytes;   // K/V bytes of one decode work unit
  float tile_bytes;   // K/V bytes of one prefill key tile (128 keys of one kv head)
  float hbm, dec_sm, pf_sm;  // bytes per ns
};

// The second stream of a device and the two events that fork it from, and join it back
// into, the caller's stream; `lock` serialises the fork/join sequence between host threads.
struct SideStream {
  cudaStream_t stream;
  cudaEvent_t fork, join;
  void* lock;  // std::mutex
};
bool side_stream_for_device(SideStream* s);
int overlap_choice();

// Launch `kernel` on `stream`, with programmatic stream serialisation (PDL) when `pdl`: it
// may then begin while the previous kernel on the stream finishes; the kernel itself calls
// pdl_wait() before touching anything an earlier kernel wrote (a no-op without PDL).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  return launch_kernel(true, kernel, grid, block, smem, stream, static_cast<Args&&>(args)...);
}

// Raises `Kernel`'s dynamic shared-memory limit to `bytes`, once per device (thread-safe:
// std::call_once); later calls return the status of that one attribute call.
template <auto Kernel>
cudaError_t set_smem_once(int bytes) {
  constexpr int kDevices = 64;
  static std::once_flag once[kDevices];
  static cudaError_t status[kDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kDevices) return cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  std::call_once(once[dev], [bytes, dev] {
    status[dev] = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  });
  return status[dev];
}

// Records the caller's timing event around a kernel launch when one is registered
// (pkv_set_kernel_events); `after` selects the stop event.
void record_kernel_event(int which, bool after, cudaStream_t stream);
int decode_ctas_for_device();
int decode_kernel_choice();
int fault_injection_choice();
int prefill_kernel_choice();

}  // namespace pkv
