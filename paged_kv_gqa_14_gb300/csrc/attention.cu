// paged_attention: work planner, decode split-K, prefill-chunk tiles and split merge.
//
// Launch sequence on the caller's stream (no host synchronisation; every grid size comes
// from tensor shapes only):
//   1. plan_kernel      (1 CTA)   classify spans, build the decode unit ranges and the
//                                 prefill tile list in the workspace
//   2. prefill kernel   (persistent) causal varlen tiles for spans longer than one row
//   3. decode kernel    (1 CTA/SM) split-K over page groups for spans of one row
//      ... and the CTA that writes the last split state of a sequence cut by a CTA boundary
//      merges that sequence's states (the split merge runs inside the decode kernel)
// Every kernel is launched with programmatic dependent launch, so each one's launch and
// prologue overlap the previous kernel's tail.  Right after the step's kv_append a caller may
// let the planner do its arithmetic while the append runs (PKV_ATTN_PLAN_EARLY) and, further,
// publish the plan through a ready word at once, so that the tensor-core decode copies the
// pages holding no new key before the append has finished (PKV_ATTN_STREAM_EARLY).  A batch
// with prefill spans instead runs
// the prefill kernel on a second stream, forked after the planner and joined back before
// the call returns, at the same time as the decode: the planner gives the prefill P of
// the SMs and spreads the decode units over the rest (SplitArgs in internal.h).
#include <cstring>
#include <mutex>

#include "decode.cuh"
#include "decode_tc.cuh"
#include "prefill.cuh"
#include "prefill_tc.cuh"

namespace pkv {

// cuTensorMapEncodeTiled, fetched from the driver once (no link-time dependency on libcuda)
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Encodes a bf16, 128-byte-swizzled tiled tensor map, reusing the last few encodings made
// on this host thread: a serving loop passes the same pool (and often the same q buffer)
// every step, and the key holds every input of the encoding, so a hit is the same map.
bool encode_bf16_sw128(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                       const cuuint64_t* strides, const cuuint32_t* box) {
  struct Key {
    const void* base;
    int rank;
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5];
  };
  struct Entry {
    Key key;
    CUtensorMap map;
    bool valid;
  };
  constexpr int kEntries = 8;
  thread_local Entry cache[kEntries] = {};
  thread_local int next = 0;
  if (rank < 1 || rank > 5) return false;
  Key key;
  memset(&key, 0, sizeof(key));
  key.base = base;
  key.rank = rank;
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
    if (i + 1 < rank) key.strides[i] = strides[i];
  }
  for (Entry& e : cache)
    if (e.valid && memcmp(&e.key, &key, sizeof(Key)) == 0) {
      *m = e.map;
      return true;
    }
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  if (fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims,
         strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache[next].key = key;
  cache[next].map = *m;
  cache[next].valid = true;
  next = (next + 1) % kEntries;
  return true;
}

// The pool [num_blocks][block_size][Hkv][d] as a 4-D tensor {d, Hkv, block_size, num_blocks};
// a box is all block_size token rows x 64 dims of one kv head in one block, 128-byte swizzled
// (the tcgen05 prefill's K/V tiles).
bool make_pool_map(CUtensorMap* m, const void* base, int64_t num_blocks, int bs_log2, int hkv, int D) {
  const cuuint64_t bs = cuuint64_t(1) << bs_log2;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(hkv), bs,
                              static_cast<cuuint64_t>(num_blocks > 0 ? num_blocks : 1)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(hkv) * D * 2,
                                 bs * hkv * D * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(bs), 1};
  return encode_bf16_sw128(m, base, 4, dims, strides, box);
}

namespace {

constexpr int kPlanThreads = 1024;
static_assert(kPlanThreads == kSmallPlanMaxSeqs, "the small planner takes one sequence per thread");

struct Int3 {
  int a, b, c;
};

// Block-wide exclusive scan of three counters at once.  `tot` receives the block totals.
__device__ Int3 block_scan3(Int3 v, Int3& tot, int* sm /* [3 * 32] */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  Int3 x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int ya = __shfl_up_sync(0xffffffffu, x.a, off);
    const int yb = __shfl_up_sync(0xffffffffu, x.b, off);
    const int yc = __shfl_up_sync(0xffffffffu, x.c, off);
    if (lane >= off) {
      x.a += ya;
      x.b += yb;
      x.c += yc;
    }
  }
  if (lane == 31) {
    sm[warp * 3 + 0] = x.a;
    sm[warp * 3 + 1] = x.b;
    sm[warp * 3 + 2] = x.c;
  }
  __syncthreads();
  if (warp == 0) {
    Int3 w = {0, 0, 0};
    if (lane < nwarps) w = {sm[lane * 3], sm[lane * 3 + 1], sm[lane * 3 + 2]};
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int ya = __shfl_up_sync(0xffffffffu, w.a, off);
      const int yb = __shfl_up_sync(0xffffffffu, w.b, off);
      const int yc = __shfl_up_sync(0xffffffffu, w.c, off);
      if (lane >= off) {
        w.a += ya;
        w.b += yb;
        w.c += yc;
      }
    }
    if (lane < nwarps) {
      sm[lane * 3 + 0] = w.a;
      sm[lane * 3 + 1] = w.b;
      sm[lane * 3 + 2] = w.c;
    }
  }
  __syncthreads();
  Int3 base = {0, 0, 0};
  if (warp > 0) base = {sm[(warp - 1) * 3], sm[(warp - 1) * 3 + 1], sm[(warp - 1) * 3 + 2]};
  tot = {sm[(nwarps - 1) * 3], sm[(nwarps - 1) * 3 + 1], sm[(nwarps - 1) * 3 + 2]};
  __syncthreads();
  return {base.a + x.a - v.a, base.b + x.b - v.b, base.c + x.c - v.c};
}

// Span classification and work lists ("09 -- Mini Inference Engine (The Capstone)",
// "Week 3 -- Continuous batching": prefill and decode sequences mixed in one batch).
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t* __restrict__ qsl,
                                                            const int32_t* __restrict__ ctxl,
                                                            int num_seqs, int64_t num_tokens,
                                                            int64_t max_ctx, int pps,
                                                            int decode_ctas, int tile_q, Plan plan,
                                                            int64_t max_tiles, SplitArgs split,
                                                            int rows_in_decode, unsigned int* err) {
  __shared__ int sm[3 * 32];
  __shared__ int carry[3];
  __shared__ unsigned long long pf_keytiles;  // 128-key tiles over all prefill q tiles (one kv head)
  __shared__ int pf_maxtile;                  // the most key tiles of one q tile
  __shared__ unsigned long long best;         // (cost bits << 32) | prefill CTAs
  if (threadIdx.x == 0) {
    carry[0] = carry[1] = carry[2] = 0;
    pf_keytiles = 0;
    pf_maxtile = 0;
    best = ~0ull;
  }
  __syncthreads();
  pdl_wait();  // the workspace may still be read by the previous call's kernels until now
  pdl_trigger();
  for (int base = 0; base < num_seqs; base += kPlanThreads) {
    const int b = base + threadIdx.x;
    Int3 v = {0, 0, 0};
    if (b < num_seqs) {
      const int s0 = qsl[b], s1 = qsl[b + 1];
      const int ctx = ctxl[b];
      const int span = s1 - s0;
      bool ok = s0 >= 0 && span >= 0 && s1 <= num_tokens;
      if (!ok) {
        raise_error(err, PKV_DEVERR_SPAN);
      } else if (span > 0) {
        if (ctx < span) {
          raise_error(err, PKV_DEVERR_SPAN);
          ok = false;
        } else if (static_cast<int64_t>(ctx) > max_ctx) {  // more keys than the table row maps
          raise_error(err, PKV_DEVERR_CONTEXT);
          ok = false;
        }
      }
      if (ok && (span == 1 || (span > 1 && rows_in_decode))) {
        // one decode entry per row: row r sees keys 0 .. ctx - span + r
        v.a = span;
        for (int r = 0; r < span; ++r) v.b += ceil_div(ceil_div(ctx - span + r + 1, kPageTokens), pps);
      }
      if (ok && span > 1 && !rows_in_decode) {
        v.c = ceil_div(span, tile_q);
        if (split.on) {  // keys [0, kv_end) of q tile j are read in 128-key tiles
          unsigned long long sum = 0;
          int mx = 0;
          for (int j = 0; j < v.c; ++j) {
            const int nk = ceil_div(ctx - span + min((j + 1) * tile_q, span), 128);
            sum += static_cast<unsigned long long>(nk);
            mx = max(mx, nk);
          }
          atomicAdd(&pf_keytiles, sum);
          atomicMax(&pf_maxtile, mx);
        }
      }
    }
    Int3 tot;
    Int3 ex = block_scan3(v, tot, sm);
    ex.a += carry[0];
    ex.b += carry[1];
    ex.c += carry[2];
    if (v.a) {
      const int ctx = ctxl[b], s0 = qsl[b];
      int unit = ex.b;
      for (int r = 0; r < v.a; ++r) {
        const int ctx_r = ctx - v.a + r + 1;
        plan.dec_seq[ex.a + r] = b;
        plan.dec_count[ex.a + r] = 0;
        plan.dec_unit[ex.a + r] = unit;
        plan.dec_ctx[ex.a + r] = ctx_r;
        plan.dec_tq[ex.a + r] = s0 + r;
        unit += ceil_div(ceil_div(ctx_r, kPageTokens), pps);
      }
    }
    for (int j = 0; j < v.c; ++j) {
      if (ex.c + j < max_tiles) {
        plan.pf_seq[ex.c + j] = b;
        plan.pf_tile[ex.c + j] = j;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      carry[0] += tot.a;
      carry[1] += tot.b;
      carry[2] += tot.c;
    }
    __syncthreads();
  }
  const int n_dec = carry[0];
  const int U = carry[1];
  const int n_tiles = static_cast<int>(min(static_cast<int64_t>(carry[2]), max_tiles));
  // prefill CTAs that take items, and the decode CTAs the units are spread over
  int pn = split.pf_grid;  // serial order: every launched prefill CTA
  int dctas = decode_ctas;
  if (split.on) {
    const int64_t items = static_cast<int64_t>(n_tiles) * split.hkv;
    int hi = static_cast<int>(min(static_cast<int64_t>(split.pf_grid), items));
    if (U > 0) hi = min(hi, split.sms - 1);
    if (hi <= 0) {
      pn = 0;
    } else if (U == 0) {
      pn = hi;
    } else {
      // the share minimising max(decode time on sms - p SMs, prefill time on p SMs)
      const float kt = static_cast<float>(pf_keytiles) * static_cast<float>(split.hkv);
      const float dec_bytes = static_cast<float>(U) * split.unit_bytes;
      for (int p = 1 + static_cast<int>(threadIdx.x); p <= hi; p += kPlanThreads) {
        const float t_dec = dec_bytes / fminf(split.hbm, static_cast<float>(split.sms - p) * split.dec_sm);
        const float t_pf = fmaxf(kt / static_cast<float>(p), static_cast<float>(pf_maxtile)) * split.tile_bytes /
                           split.pf_sm;
        const unsigned long long key =
            (static_cast<unsigned long long>(__float_as_uint(fmaxf(t_dec, t_pf))) << 32) | static_cast<unsigned>(p);
        atomicMin(&best, key);
      }
      __syncthreads();
      pn = static_cast<int>(best & 0xffffffffu);
    }
    if (U > 0) dctas = split.sms - pn;
  }
  const int W = max(1, ceil_div(U, max(1, dctas)));
  if (threadIdx.x == 0) plan.dec_unit[n_dec] = U;
  __syncthreads();

  // split pieces per decode sequence and the first partial slot of each
  __shared__ int carry2;
  if (threadIdx.x == 0) carry2 = 0;
  __syncthreads();
  for (int base = 0; base < n_dec; base += kPlanThreads) {
    const int i = base + threadIdx.x;
    Int3 v = {0, 0, 0};
    if (i < n_dec) {
      const int u0 = plan.dec_unit[i], u1 = plan.dec_unit[i + 1];
      v.a = (u1 - 1) / W - u0 / W + 1;
    }
    Int3 tot;
    const Int3 ex = block_scan3(v, tot, sm);
    if (i < n_dec) {
      plan.dec_slot[i] = ex.a + carry2;
      plan.dec_chunks[i] = v.a;
      // the start records of the decode CTAs whose first unit c W falls in this entry's units
      // [u0, u1)
      const int u0 = plan.dec_unit[i], u1 = plan.dec_unit[i + 1];
      const int4 r0 = make_int4(i, u0, u1, plan.dec_seq[i]);
      const int4 r1 = make_int4(plan.dec_ctx[i], plan.dec_tq[i], 0, 0);
      for (int c = ceil_div(u0, W); c * W < u1; ++c) {
        plan.cta_rec[2 * c] = r0;
        plan.cta_rec[2 * c + 1] = r1;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) carry2 += tot.a;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    plan.header[0] = n_dec;
    plan.header[1] = U;
    plan.header[2] = W;
    plan.header[3] = n_tiles;
    plan.header[4] = carry2;
    plan.header[5] = pn;
  }
}

// The same plan for a batch of at most kPlanThreads sequences, one thread per sequence,
// computed in registers and shared memory first and written to the workspace at the end.
// With `early` the arithmetic runs before the wait on the previous kernel (only the inputs
// query_start_loc and context_lens are read by then; the caller vouches that the kernel
// before this call does not write them) and only the workspace writes come after it, so the
// planner's work overlaps that kernel (the step's kv_append).  Without `early` it waits
// first, like plan_kernel.
// With `stream` (which implies `early`) the workspace is written as soon as the plan is known,
// and header[kPlanReadyWord] then tells the decode it may start streaming pages (cleared
// before this kernel lets the decode launch, set after every other workspace write): 1 when
// each decode entry's new keys all lie in its last 16-token page (every entry is a span of
// one token), 2 when some entry is a row of a longer span.  The kernel still waits on the
// previous kernel before it ends, so work that waits for its end waits for that kernel too.
// (`stream` 2, a test-only fault: everything as with 1 but the word is never published, so
// the decode's bounded polls run out and it falls back to waiting for this kernel's end.)
__global__ void __launch_bounds__(kPlanThreads) plan_kernel_small(const int32_t* __restrict__ qsl,
                                                                  const int32_t* __restrict__ ctxl,
                                                                  int num_seqs, int64_t num_tokens,
                                                                  int64_t max_ctx, int pps, int decode_ctas,
                                                                  int tile_q, Plan plan, int64_t max_tiles,
                                                                  SplitArgs split, int rows_in_decode, int early,
                                                                  int stream, unsigned int* err) {
  __shared__ int sm[3 * 32];
  __shared__ unsigned long long pf_keytiles;  // 128-key tiles over all prefill q tiles (one kv head)
  __shared__ int pf_maxtile;                  // the most key tiles of one q tile
  __shared__ unsigned long long best;         // (cost bits << 32) | prefill CTAs
  if (threadIdx.x == 0) {
    pf_keytiles = 0;
    pf_maxtile = 0;
    best = ~0ull;
  }
  if (stream) {
    if (threadIdx.x == 0) {
      plan.header[kPlanReadyWord] = 0;
      __threadfence();
    }
    __syncthreads();
    pdl_trigger();  // the decode may start; it reads nothing of the plan before the ready word
  } else if (early) {
    pdl_trigger();  // the decode may start its prologue; it waits for this kernel's end
  } else {
    pdl_wait();  // the workspace may still be read by the previous call's kernels until now
    pdl_trigger();
  }
  __syncthreads();
  // this thread's sequence: decode entries (a), work units (b), prefill q tiles (c)
  const int b = threadIdx.x;
  int s0 = 0, span = 0, ctx = 0;
  Int3 v = {0, 0, 0};
  if (b < num_seqs) {
    s0 = qsl[b];
    const int s1 = qsl[b + 1];
    ctx = ctxl[b];
    span = s1 - s0;
    bool ok = s0 >= 0 && span >= 0 && s1 <= num_tokens;
    if (!ok) {
      raise_error(err, PKV_DEVERR_SPAN);
    } else if (span > 0) {
      if (ctx < span) {
        raise_error(err, PKV_DEVERR_SPAN);
        ok = false;
      } else if (static_cast<int64_t>(ctx) > max_ctx) {  // more keys than the table row maps
        raise_error(err, PKV_DEVERR_CONTEXT);
        ok = false;
      }
    }
    if (ok && (span == 1 || (span > 1 && rows_in_decode))) {
      // one decode entry per row: row r sees keys 0 .. ctx - span + r
      v.a = span;
      for (int r = 0; r < span; ++r) v.b += ceil_div(ceil_div(ctx - span + r + 1, kPageTokens), pps);
    }
    if (ok && span > 1 && !rows_in_decode) {
      v.c = ceil_div(span, tile_q);
      if (split.on) {  // keys [0, kv_end) of q tile j are read in 128-key tiles
        unsigned long long sum = 0;
        int mx = 0;
        for (int j = 0; j < v.c; ++j) {
          const int nk = ceil_div(ctx - span + min((j + 1) * tile_q, span), 128);
          sum += static_cast<unsigned long long>(nk);
          mx = max(mx, nk);
        }
        atomicAdd(&pf_keytiles, sum);
        atomicMax(&pf_maxtile, mx);
      }
    }
  }
  Int3 tot;
  const Int3 ex = block_scan3(v, tot, sm);
  const int n_dec = tot.a;
  const int U = tot.b;
  const int n_tiles = static_cast<int>(min(static_cast<int64_t>(tot.c), max_tiles));
  // prefill CTAs that take items, and the decode CTAs the units are spread over (as plan_kernel)
  int pn = split.pf_grid;
  int dctas = decode_ctas;
  if (split.on) {
    const int64_t items = static_cast<int64_t>(n_tiles) * split.hkv;
    int hi = static_cast<int>(min(static_cast<int64_t>(split.pf_grid), items));
    if (U > 0) hi = min(hi, split.sms - 1);
    if (hi <= 0) {
      pn = 0;
    } else if (U == 0) {
      pn = hi;
    } else {
      const float kt = static_cast<float>(pf_keytiles) * static_cast<float>(split.hkv);
      const float dec_bytes = static_cast<float>(U) * split.unit_bytes;
      for (int p = 1 + static_cast<int>(threadIdx.x); p <= hi; p += kPlanThreads) {
        const float t_dec = dec_bytes / fminf(split.hbm, static_cast<float>(split.sms - p) * split.dec_sm);
        const float t_pf = fmaxf(kt / static_cast<float>(p), static_cast<float>(pf_maxtile)) * split.tile_bytes /
                           split.pf_sm;
        const unsigned long long key =
            (static_cast<unsigned long long>(__float_as_uint(fmaxf(t_dec, t_pf))) << 32) | static_cast<unsigned>(p);
        atomicMin(&best, key);
      }
      __syncthreads();
      pn = static_cast<int>(best & 0xffffffffu);
    }
    if (U > 0) dctas = split.sms - pn;
  }
  const int W = max(1, ceil_div(U, max(1, dctas)));
  // split pieces of this thread's decode entries: the decode CTAs touching each entry
  Int3 pc = {0, 0, 0};
  {
    int unit = ex.b;
    for (int r = 0; r < v.a; ++r) {
      const int u1 = unit + ceil_div(ceil_div(ctx - v.a + r + 1, kPageTokens), pps);
      pc.a += (u1 - 1) / W - unit / W + 1;
      unit = u1;
    }
  }
  Int3 ptot;
  const Int3 pex = block_scan3(pc, ptot, sm);

  // a decode entry that is one row of a longer span has new keys before its last page
  const int long_rows = __syncthreads_or(v.a > 1);
  if (early && !stream) pdl_wait();  // from here on the workspace is written
  {
    int unit = ex.b, slot = pex.a;
    for (int r = 0; r < v.a; ++r) {
      const int i = ex.a + r;
      const int ctx_r = ctx - v.a + r + 1;
      const int u1 = unit + ceil_div(ceil_div(ctx_r, kPageTokens), pps);
      const int pieces = (u1 - 1) / W - unit / W + 1;
      plan.dec_seq[i] = b;
      plan.dec_count[i] = 0;
      plan.dec_unit[i] = unit;
      plan.dec_ctx[i] = ctx_r;
      plan.dec_tq[i] = s0 + r;
      plan.dec_slot[i] = slot;
      plan.dec_chunks[i] = pieces;
      // the start records of the decode CTAs whose first unit c W falls in [unit, u1)
      const int4 r0 = make_int4(i, unit, u1, b);
      const int4 r1 = make_int4(ctx_r, s0 + r, 0, 0);
      for (int c = ceil_div(unit, W); c * W < u1; ++c) {
        plan.cta_rec[2 * c] = r0;
        plan.cta_rec[2 * c + 1] = r1;
      }
      slot += pieces;
      unit = u1;
    }
  }
  for (int j = 0; j < v.c; ++j) {
    if (ex.c + j < max_tiles) {
      plan.pf_seq[ex.c + j] = b;
      plan.pf_tile[ex.c + j] = j;
    }
  }
  if (threadIdx.x == 0) {
    plan.dec_unit[n_dec] = U;
    plan.header[0] = n_dec;
    plan.header[1] = U;
    plan.header[2] = W;
    plan.header[3] = n_tiles;
    plan.header[4] = ptot.a;
    plan.header[5] = pn;
  }
  if (stream) {
    __syncthreads();  // every thread's workspace writes are done
    if (threadIdx.x == 0 && stream == 1) {
      __threadfence();
      st_release_gpu(plan.header + kPlanReadyWord, long_rows ? 2 : 1);
    }
    pdl_wait();  // this kernel ends after the previous one
  }
}

template <int D, int G>
cudaError_t launch_decode(const AttnArgs& a, cudaStream_t stream) {
  using C = DecodeCfg<D, G>;
  if (const cudaError_t e = set_smem_once<decode_splitk_kernel<D, G>>(C::kSmemBytes); e != cudaSuccess) return e;
  DecodeParams p;
  p.q = static_cast<const bf16*>(a.q);
  p.q_st = a.q_st;
  p.q_sh = a.q_sh;
  p.k_cache = static_cast<const bf16*>(a.k_cache);
  p.v_cache = static_cast<const bf16*>(a.v_cache);
  p.num_blocks = a.num_blocks;
  p.bs_log2 = a.bs_log2;
  p.block_tables = a.block_tables;
  p.bt_stride = a.bt_stride;
  p.context_lens = a.context_lens;
  p.qsl = a.qsl;
  p.out = static_cast<bf16*>(a.out);
  p.o_st = a.o_st;
  p.o_sh = a.o_sh;
  p.hkv = a.hkv;
  p.hq = a.hq;
  p.qscale = a.scale * 1.4426950408889634f;
  p.plan = a.plan;
  p.err = a.err;
  p.fault_no_copies = 0;
  p.stream_early = 0;  // this kernel waits for the whole plan
  record_kernel_event(PKV_KERNEL_DECODE, false, stream);
  const cudaError_t e = launch_pdl(decode_splitk_kernel<D, G>, dim3(a.decode_ctas), dim3((kDecodeWarps + 1) * 32),
                                   C::kSmemBytes, stream, p);
  record_kernel_event(PKV_KERNEL_DECODE, true, stream);
  return e;
}

template <int D>
cudaError_t launch_decode_g(const AttnArgs& a, cudaStream_t stream) {
  switch (a.hq / a.hkv) {
    case 1: return launch_decode<D, 1>(a, stream);
    case 2: return launch_decode<D, 2>(a, stream);
    case 3: return launch_decode<D, 3>(a, stream);
    case 4: return launch_decode<D, 4>(a, stream);
    case 5: return launch_decode<D, 5>(a, stream);
    case 6: return launch_decode<D, 6>(a, stream);
    case 7: return launch_decode<D, 7>(a, stream);
    case 8: return launch_decode<D, 8>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

// q [T][Hq][d] as a 3-D tensor {d, Hq, T}; a box is 128 token rows x 64 dims of one head.
bool make_q_map(CUtensorMap* m, const AttnArgs& a) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.head_dim), static_cast<cuuint64_t>(a.hq),
                              static_cast<cuuint64_t>(a.num_tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.q_sh) * 2, static_cast<cuuint64_t>(a.q_st) * 2};
  // a box is the G heads of one kv head's group x P consecutive tokens x 64 dims
  const int g = a.hq / a.hkv;
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(kTcPrefillRows / g)};
  return encode_bf16_sw128(m, a.q, 3, dims, strides, box);
}

bool make_prefill_tc_params(const AttnArgs& a, PrefillTcParams* P) {
  if (a.q_sh <= 0 || a.q_st <= 0) return false;
  if (!make_q_map(&P->tmap_q, a) ||
      !make_pool_map(&P->tmap_k, a.k_cache, a.num_blocks, a.bs_log2, a.hkv, a.head_dim) ||
      !make_pool_map(&P->tmap_v, a.v_cache, a.num_blocks, a.bs_log2, a.hkv, a.head_dim))
    return false;
  P->p = make_prefill_params(a);
  P->group = a.hq / a.hkv;
  P->prows = kTcPrefillRows / P->group;
  return true;
}

// CTAs the tcgen05 prefill is launched with: one per SM, at most one per item.
int64_t prefill_tc_grid(const AttnArgs& a, int prows) {
  const int64_t max_items = (a.num_tokens / prows + a.num_seqs + 1) * a.hkv;
  const int64_t cap = device_sm_count();
  return max_items < cap ? max_items : cap;
}

template <int D>
cudaError_t launch_prefill_tc(const AttnArgs& a, const PrefillTcParams& P, cudaStream_t stream, bool pdl) {
  using C = PrefillTcCfg<D>;
  if (const cudaError_t e = set_smem_once<prefill_tc_kernel<D>>(C::kSmemBytes); e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(prefill_tc_grid(a, P.prows));
  record_kernel_event(PKV_KERNEL_PREFILL, false, stream);
  const cudaError_t e = launch_kernel(pdl, prefill_tc_kernel<D>, dim3(grid), dim3(256), C::kSmemBytes, stream, P);
  record_kernel_event(PKV_KERNEL_PREFILL, true, stream);
  return e;
}

}  // namespace

// The pool viewed head-major for the decode, {d, block_size, Hkv, num_blocks} with strides
// (a row, a head, a block); a box is 64 dims x min(block_size, 16) rows x all kv heads of one
// block, 128-byte swizzled, landing as [kv head][rows][128 bytes].
bool make_pool_map_heads(CUtensorMap* m, const void* base, int64_t num_blocks, int bs_log2, int hkv, int D) {
  const cuuint64_t bs = cuuint64_t(1) << bs_log2;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), bs, static_cast<cuuint64_t>(hkv),
                              static_cast<cuuint64_t>(num_blocks > 0 ? num_blocks : 1)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(hkv) * D * 2, static_cast<cuuint64_t>(D) * 2,
                                 bs * hkv * D * 2};
  const cuuint32_t box[4] = {64, bs < 16 ? static_cast<cuuint32_t>(bs) : 16u, static_cast<cuuint32_t>(hkv), 1};
  return encode_bf16_sw128(m, base, 4, dims, strides, box);
}

cudaError_t launch_paged_attention(const AttnArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.num_tokens == 0) return cudaSuccess;
  const int pps = kDecodeWarps / a.hkv;
  // prefill arithmetic: tcgen05 (128-row tiles) when chosen and its q tensor map encodes,
  // else mma.sync (64-row tiles)
  PrefillTcParams tcp;
  const bool use_tc = a.prefill_kernel == 2 && make_prefill_tc_params(a, &tcp);
  const int tile_q = use_tc ? kTcPrefillRows / (a.hq / a.hkv) : kPrefillTileQ;
  const int sms = device_sm_count();
  const int64_t pf_grid = use_tc ? prefill_tc_grid(a, tcp.prows) : prefill_mma_grid(a);
  // Prefill beside the decode: only with spans of two or more tokens (more tokens than
  // sequences), the tcgen05 tiles (one CTA per SM) and the default one decode CTA per SM, on
  // the caller's second stream (with its fork/join events) or else the library's own.
  SideStream side{};
  bool split = a.overlap && use_tc && a.num_tokens > a.num_seqs && a.decode_ctas == sms && sms > 1;
  const bool own_side = split && a.side_stream == nullptr;
  if (split && !own_side) {
    side.stream = a.side_stream;
    side.fork = a.fork_event;
    side.join = a.join_event;
  } else if (own_side) {
    split = side_stream_for_device(&side);
  }
  // The library's side stream is shared by every caller on the device; its use, from this
  // check to the join, is serialised by a host mutex.  Through the fork event it joins a graph
  // capture of the caller's stream and stays in that capture until the capture ends, so it
  // is taken only when no capture holds it, or when the capture holding it is this call's;
  // otherwise this call runs in the serial order.
  std::unique_lock<std::mutex> hold;
  if (split && own_side) {
    hold = std::unique_lock<std::mutex>(*static_cast<std::mutex*>(side.lock));
    cudaStreamCaptureStatus st_side = cudaStreamCaptureStatusNone, st_call = cudaStreamCaptureStatusNone;
    unsigned long long id_side = 0, id_call = 0;
    if (cudaStreamGetCaptureInfo(side.stream, &st_side, &id_side) != cudaSuccess ||
        cudaStreamGetCaptureInfo(stream, &st_call, &id_call) != cudaSuccess) {
      split = false;
    } else if (st_side != cudaStreamCaptureStatusNone &&
               !(st_side == cudaStreamCaptureStatusActive && st_call == cudaStreamCaptureStatusActive &&
                 id_side == id_call)) {
      split = false;
    }
    if (!split) hold.unlock();
  }
  SplitArgs sp{};
  sp.on = split ? 1 : 0;
  sp.sms = sms;
  sp.pf_grid = static_cast<int>(pf_grid);
  sp.hkv = a.hkv;
  sp.unit_bytes = static_cast<float>(kDecodeWarps) * kPageTokens * a.head_dim * 4.f;  // pps x hkv = 8 pages of K and V
  sp.tile_bytes = 128.f * a.head_dim * 4.f;
  sp.hbm = kSplitHbmBytesPerNs;
  sp.dec_sm = kSplitDecodeSmBytesPerNs;
  sp.pf_sm = split_prefill_sm_bytes_per_ns(a.bs_log2);
  record_kernel_event(PKV_KERNEL_PLAN, false, stream);
  // With no more tokens than sequences a prefill span is rare (it needs empty spans beside it):
  // no prefill kernel is launched (its idle CTAs would hold the SMs between the planner and
  // the decode), and the rows of such a span become decode entries.
  const bool rows_in_decode = a.num_tokens <= a.num_seqs;
  // up to kPlanThreads sequences: one thread each, the workspace written at the end (and, with
  // plan_early, the arithmetic done before the wait on the previous kernel)
  cudaError_t e =
      a.num_seqs <= kPlanThreads
          ? launch_pdl(plan_kernel_small, dim3(1), dim3(kPlanThreads), 0, stream, a.qsl, a.context_lens,
                       static_cast<int>(a.num_seqs), a.num_tokens, a.max_blocks << a.bs_log2, pps, a.decode_ctas,
                       tile_q, a.plan, a.max_tiles, sp, rows_in_decode ? 1 : 0, a.plan_early ? 1 : 0,
                       a.stream_early ? (a.fault == PKV_FAULT_PLAN_NO_READY ? 2 : 1) : 0, a.err)
          : launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, a.qsl, a.context_lens,
                       static_cast<int>(a.num_seqs), a.num_tokens, a.max_blocks << a.bs_log2, pps, a.decode_ctas,
                       tile_q, a.plan, a.max_tiles, sp, rows_in_decode ? 1 : 0, a.err);
  record_kernel_event(PKV_KERNEL_PLAN, true, stream);
  if (e != cudaSuccess) return e;
  auto prefill = [&](cudaStream_t s, bool pdl) -> cudaError_t {
    if (use_tc)
      return (a.head_dim == 128) ? launch_prefill_tc<128>(a, tcp, s, pdl) : launch_prefill_tc<64>(a, tcp, s, pdl);
    return (a.head_dim == 128) ? launch_prefill<128>(a, s, pdl) : launch_prefill<64>(a, s, pdl);
  };
  auto decode = [&]() -> cudaError_t {
    const int kind = a.decode_kernel != 0 ? a.decode_kernel : (a.hq / a.hkv >= kTensorDecodeMinGroup ? 2 : 1);
    if (kind == 2) {
      switch (a.bs_log2) {  // one compiled instance per block size (decode_tc.cu)
        case 3: return launch_decode_tc_bs8(a, stream);
        case 4: return launch_decode_tc_bs16(a, stream);
        case 5: return launch_decode_tc_bs32(a, stream);
        case 6: return launch_decode_tc_bs64(a, stream);
        case 7: return launch_decode_tc_bs128(a, stream);
        default: return cudaErrorInvalidValue;
      }
    }
    return (a.head_dim == 128) ? launch_decode_g<128>(a, stream) : launch_decode_g<64>(a, stream);
  };
  if (!split) {
    if (!rows_in_decode && (e = prefill(stream, true)) != cudaSuccess) return e;
    return decode();
  }
  // fork after the planner, decode here, prefill on the side stream, join before returning
  if ((e = cudaEventRecord(side.fork, stream)) != cudaSuccess) return e;
  if ((e = decode()) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(side.stream, side.fork, 0)) != cudaSuccess) return e;
  if ((e = prefill(side.stream, false)) != cudaSuccess) return e;
  if ((e = cudaEventRecord(side.join, side.stream)) != cudaSuccess) return e;
  return cudaStreamWaitEvent(stream, side.join, 0);
}

// ------------------------------------------------------------------ workspace layout
static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

PlanSizes plan_sizes(int64_t num_tokens, int64_t num_seqs, int64_t num_q_heads, int64_t head_dim,
                     int64_t decode_ctas) {
  PlanSizes s{};
  s.num_seqs = num_seqs;
  s.num_tokens = num_tokens;
  s.num_q_heads = num_q_heads;
  s.head_dim = head_dim;
  s.decode_ctas = decode_ctas;
  s.max_tiles = num_tokens / kMinPrefillTileQ + num_seqs + 1;
  s.max_slots = num_seqs + decode_ctas;
  size_t off = 0;
  s.off_header = off;
  off = align256(off + 16 * sizeof(int));
  s.off_dec_seq = off;
  off = align256(off + num_seqs * sizeof(int));
  s.off_dec_unit = off;
  off = align256(off + (num_seqs + 1) * sizeof(int));
  s.off_dec_slot = off;
  off = align256(off + num_seqs * sizeof(int));
  s.off_dec_chunks = off;
  off = align256(off + num_seqs * sizeof(int));
  s.off_dec_count = off;
  off = align256(off + num_seqs * sizeof(int));
  s.off_dec_ctx = off;
  off = align256(off + num_seqs * sizeof(int));
  s.off_dec_tq = off;
  off = align256(off + num_seqs * sizeof(int));
  s.off_cta_rec = off;
  off = align256(off + decode_ctas * 2 * sizeof(int4));
  s.off_pf_seq = off;
  off = align256(off + s.max_tiles * sizeof(int));
  s.off_pf_tile = off;
  off = align256(off + s.max_tiles * sizeof(int));
  s.off_part_ml = off;
  off = align256(off + s.max_slots * num_q_heads * 2 * sizeof(float));
  s.off_part_acc = off;
  off = align256(off + s.max_slots * num_q_heads * head_dim * sizeof(float));
  s.total = off;
  return s;
}

Plan plan_view(void* workspace, const PlanSizes& s) {
  char* w = static_cast<char*>(workspace);
  Plan p;
  p.header = reinterpret_cast<int*>(w + s.off_header);
  p.dec_seq = reinterpret_cast<int*>(w + s.off_dec_seq);
  p.dec_unit = reinterpret_cast<int*>(w + s.off_dec_unit);
  p.dec_slot = reinterpret_cast<int*>(w + s.off_dec_slot);
  p.dec_chunks = reinterpret_cast<int*>(w + s.off_dec_chunks);
  p.dec_count = reinterpret_cast<int*>(w + s.off_dec_count);
  p.dec_ctx = reinterpret_cast<int*>(w + s.off_dec_ctx);
  p.dec_tq = reinterpret_cast<int*>(w + s.off_dec_tq);
  p.cta_rec = reinterpret_cast<int4*>(w + s.off_cta_rec);
  p.pf_seq = reinterpret_cast<int*>(w + s.off_pf_seq);
  p.pf_tile = reinterpret_cast<int*>(w + s.off_pf_tile);
  p.part_ml = reinterpret_cast<float*>(w + s.off_part_ml);
  p.part_acc = reinterpret_cast<float*>(w + s.off_part_acc);
  return p;
}

}  // namespace pkv
