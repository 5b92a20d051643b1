// Decode split-K kernel: one query row per sequence ("mini_engine" README, "Where the gap
// comes from": attention over the paged blocks is the memory traffic that dominates a
// decode step; "09 -- Mini Inference Engine (The Capstone)", "Week 4 -- Paged KV cache":
// attention reads the context through the block table).
//
// Work decomposition.  A work unit is one page group of one decode sequence: P = 8 / Hkv
// consecutive 16-token pages with all kv heads.  For a pool laid out
// [num_blocks][16][Hkv][d] a page with all heads is one contiguous run of 16*Hkv*d bf16,
// so each page of K (and of V) is ONE 1-D bulk copy (TMA, cp.async.bulk) into shared
// memory.  The planner concatenates all decode sequences' units and each persistent CTA
// (one per SM) takes an equal contiguous range of W units: the load is balanced to one
// unit whatever the length mix.  A sequence cut by a CTA boundary yields one split state
// (m, l, acc) per piece; the merge kernel combines them.
//
// Inside a CTA: warp 8 is the producer (one elected issue per page, a STAGES-deep ring of
// full/empty mbarriers); warps 0..7 consume.  Consumer warp w handles page w / Hkv of the
// unit and kv head w % Hkv for all G = Hq/Hkv query heads of the group, so every K/V page
// is read from HBM once per GQA group.  Each lane owns head_dim/32 dimensions: q.K partial
// sums for the 16 rows x G heads are reduced across the warp with a transposing butterfly
// (16G shuffles for all 16G sums), the online softmax runs in the log2 domain with the
// running max kept warp-uniform, and P.V accumulates in fp32 registers per lane.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace pkv {

struct DecodeParams {
  const bf16* q;
  int64_t q_st, q_sh;
  const bf16* k_cache;
  const bf16* v_cache;
  int64_t num_blocks;
  int bs_log2;  // log2 of the pool's block size
  const int32_t* block_tables;
  int64_t bt_stride;
  const int32_t* context_lens;
  const int32_t* qsl;
  bf16* out;
  int64_t o_st, o_sh;
  int hkv, hq;
  float qscale;  // softmax scale * log2(e)
  Plan plan;
  unsigned int* err;
  int fault_no_copies;  // test-only: the tensor-core decode's producer issues nothing
  int stream_early;     // the planner publishes header[kPlanReadyWord] (tensor-core decode only)
};

template <int D, int G>
struct DecodeCfg {
  static constexpr int DPL = D / 32;                      // head dims per lane
  static constexpr int kStageElems = kDecodeWarps * 16 * D;  // bf16 per K (or V) half of a stage
  static constexpr int kStageBytes = 2 * kStageElems * 2;
  static constexpr int kBarBytes = 256;
  static constexpr int kPbufBytes = kDecodeWarps * 16 * G * 4;
  static constexpr int kXbufBytes = (kDecodeWarps - 1) * G * (D + 2) * 4;
  static constexpr int kReserve = kBarBytes + kPbufBytes + kXbufBytes;
  static constexpr int kSmemLimit = 227 * 1024;
  static constexpr int kStagesFit = (kSmemLimit - kReserve) / kStageBytes;
  static constexpr int STAGES = kStagesFit > 4 ? 4 : kStagesFit;
  static constexpr int kSmemBytes = STAGES * kStageBytes + kReserve;
  static_assert(STAGES >= 2, "decode pipeline needs at least two stages");
  static_assert(DPL == 2 || DPL == 4, "head_dim must be 64 or 128");
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded mbarrier wait that also gives up once any thread of the CTA has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, unsigned int* err,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > (1ll << 31)) {
      *abort_flag = 1;
      raise_error(err, PKV_DEVERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Split merge (a6), run inside the decode kernel by the CTA that writes the LAST split state
// of decode sequence i: out = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k (scores are in
// the log2 domain).  Called by all consumer threads after they wrote this CTA's state.  Each
// writer publishes its state (fence) before counting itself in dec_count[i]; the CTA that
// counts last reads every state through L2 and writes the bf16 row.  No thread waits for
// another CTA, so there is no inter-CTA spin.
// `chunks` and `slot0` are the entry's dec_chunks[i] and dec_slot[i].  A thread merges
// kMergeItems float4 items (head, 4 dims) at a time and reads the pieces in groups of
// kMergeGroup: the (m, l) and acc loads of a whole group and of all its items are issued
// together, so an entry of up to kMergeGroup pieces costs one round trip to L2 per pass.
// Groups after the first are folded in with a running maximum (the online form of the same
// sum); with at most kMergeGroup pieces the sum is the plain one above, in piece order.
constexpr int kMergeItems = 1;
constexpr int kMergeGroup = 4;
template <int D>
__device__ void finish_split(const DecodeParams& p, int i, int64_t tq, int chunks, int slot0,
                             volatile int* last_flag) {
  constexpr int kThreads = kDecodeWarps * 32;
  constexpr int kQ = D / 4;
  __threadfence();
  named_bar_sync(1, kThreads);
  if (threadIdx.x == 0) *last_flag = atomicAdd(&p.plan.dec_count[i], 1) == chunks - 1;
  named_bar_sync(1, kThreads);
  if (*last_flag) {
    __threadfence();
    const int hq = p.hq;
    const int nitems = hq * kQ;
    const float NEG_INF = -__int_as_float(0x7f800000);
    for (int base = threadIdx.x; base < nitems; base += kMergeItems * kThreads) {
      float M[kMergeItems], den[kMergeItems];
      float4 num[kMergeItems];
#pragma unroll
      for (int j = 0; j < kMergeItems; ++j) {
        M[j] = NEG_INF;
        den[j] = 0.f;
        num[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int k0 = 0; k0 < chunks; k0 += kMergeGroup) {
        float2 ml[kMergeGroup][kMergeItems];
        float4 a[kMergeGroup][kMergeItems];
#pragma unroll
        for (int kk = 0; kk < kMergeGroup; ++kk) {
#pragma unroll
          for (int j = 0; j < kMergeItems; ++j) {
            const int item = base + j * kThreads;
            const int h = item / kQ;
            const int64_t sh = static_cast<int64_t>(slot0 + k0 + kk) * hq + h;
            if (k0 + kk < chunks && item < nitems) {
              ml[kk][j] = __ldcg(reinterpret_cast<const float2*>(p.plan.part_ml + sh * 2));
              a[kk][j] = __ldcg(reinterpret_cast<const float4*>(p.plan.part_acc + sh * D) + (item - h * kQ));
            } else {
              ml[kk][j] = make_float2(NEG_INF, 0.f);
              a[kk][j] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kMergeItems; ++j) {
          float Mn = M[j];
#pragma unroll
          for (int kk = 0; kk < kMergeGroup; ++kk) Mn = fmaxf(Mn, ml[kk][j].x);
          if (Mn == NEG_INF) continue;  // an item past the end (every piece holds a key)
          const float c = fast_exp2(M[j] - Mn);  // 0 on the first group
          den[j] *= c;
          num[j].x *= c;
          num[j].y *= c;
          num[j].z *= c;
          num[j].w *= c;
#pragma unroll
          for (int kk = 0; kk < kMergeGroup; ++kk) {
            const float w = fast_exp2(ml[kk][j].x - Mn);  // 0 for a piece past the entry
            den[j] = fmaf(w, ml[kk][j].y, den[j]);
            num[j].x = fmaf(w, a[kk][j].x, num[j].x);
            num[j].y = fmaf(w, a[kk][j].y, num[j].y);
            num[j].z = fmaf(w, a[kk][j].z, num[j].z);
            num[j].w = fmaf(w, a[kk][j].w, num[j].w);
          }
          M[j] = Mn;
        }
      }
#pragma unroll
      for (int j = 0; j < kMergeItems; ++j) {
        const int item = base + j * kThreads;
        if (item < nitems) {
          const int h = item / kQ;
          const int d0 = (item - h * kQ) * 4;
          const float inv = 1.f / den[j];
          uint2 o;
          o.x = pack_bf16x2(num[j].x * inv, num[j].y * inv);
          o.y = pack_bf16x2(num[j].z * inv, num[j].w * inv);
          *reinterpret_cast<uint2*>(p.out + tq * p.o_st + static_cast<int64_t>(h) * p.o_sh + d0) = o;
        }
      }
    }
  }
  named_bar_sync(1, kThreads);  // last_flag is reused by the next segment
}

// Load this lane's DPL bf16 of one row and widen to fp32.
template <int DPL>
__device__ __forceinline__ void load_row(const bf16* row, int lane, bool valid, float (&x)[DPL]) {
  if constexpr (DPL == 4) {
    uint2 w = valid ? *reinterpret_cast<const uint2*>(row + lane * 4) : make_uint2(0u, 0u);
    x[0] = bf16lo(w.x);
    x[1] = bf16hi(w.x);
    x[2] = bf16lo(w.y);
    x[3] = bf16hi(w.y);
  } else {
    uint32_t w = valid ? *reinterpret_cast<const uint32_t*>(row + lane * 2) : 0u;
    x[0] = bf16lo(w);
    x[1] = bf16hi(w);
  }
}

// One level of the transposing butterfly: the lane keeps the half of `v` selected by its
// bit `delta` and adds the partner's copy of that half.  N = number of values kept.
template <int N>
__device__ __forceinline__ void tr_level(float* v, int delta, int lane) {
  const bool upper = (lane & delta) != 0;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const float lo = v[k], hi = v[N + k];
    const float send = upper ? lo : hi;
    const float keep = upper ? hi : lo;
    v[k] = keep + __shfl_xor_sync(0xffffffffu, send, delta);
  }
}

template <int D, int G>
__global__ void __launch_bounds__((kDecodeWarps + 1) * 32, 1)
    decode_splitk_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecodeCfg<D, G>;
  constexpr int DPL = C::DPL;
  constexpr int STAGES = C::STAGES;
  extern __shared__ __align__(128) unsigned char smem[];
  bf16* stages = reinterpret_cast<bf16*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
  uint64_t* empty = full + STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STAGES);
  volatile int* last_flag = abort_flag + 2;
  float* pbuf = reinterpret_cast<float*>(smem + STAGES * C::kStageBytes + C::kBarBytes);
  float* xbuf = pbuf + kDecodeWarps * 16 * G;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecodeWarps);
    }
    fence_mbar_init();
    *abort_flag = 0;
  }
  pdl_wait();  // the plan is written by the planner kernel
  pdl_trigger();
  const int* hdr = p.plan.header;
  const int U = hdr[1];
  const int W = hdr[2];
  // this CTA's start record from the planner, read alongside the header: the decode entry
  // holding its first unit, that entry's unit range, sequence, context and query row
  // (meaningless, and unused, for a CTA without units)
  const int4 rec0 = p.plan.cta_rec[2 * blockIdx.x];
  const int4 rec1 = p.plan.cta_rec[2 * blockIdx.x + 1];
  const int i_first = rec0.x;
  const int ubeg = blockIdx.x * W;
  const int uend = min(U, ubeg + W);
  if (ubeg >= uend) return;  // CTA-uniform
  const int* dec_unit = p.plan.dec_unit;
  __syncthreads();  // barrier initialisation visible to every warp

  const int hkv = p.hkv;
  const int pps = kDecodeWarps / hkv;
  const int64_t page_elems = static_cast<int64_t>(16) * hkv * D;
  const uint32_t page_bytes = static_cast<uint32_t>(page_elems * 2);

  if (warp == kDecodeWarps) {
    // ------------------------------------------------------------------ producer warp
    const uint64_t pol = l2_policy_evict_first();
    int i = i_first;
    int ustart = rec0.y, unext = rec0.z;
    int b = rec0.w;
    int ctx = rec1.x;
    int npages = ceil_div(ctx, 16);
    const int sh = p.bs_log2;
    const int bmask = (1 << sh) - 1;
    const int piece_rows = sh >= 4 ? 16 : 8;  // rows of one contiguous copy
    const int64_t row_elems = static_cast<int64_t>(hkv) * D;
    int it = 0;
    for (int u = ubeg; u < uend; ++u, ++it) {
      while (u >= unext) {
        ++i;
        ustart = unext;
        unext = dec_unit[i + 1];
        b = p.plan.dec_seq[i];
        ctx = p.plan.dec_ctx[i];
        npages = ceil_div(ctx, 16);
      }
      const int pg0 = (u - ustart) * pps;
      const int npg = min(pps, npages - pg0);
      const int s = it % STAGES;
      if (it >= STAGES && !wait_or_abort(&empty[s], ((it / STAGES) - 1) & 1, p.err, abort_flag)) break;
      // with 8-token blocks the last page's second half is not copied when it lies past the
      // context (its block may not exist); the consumers never read those rows
      const bool tail_half = piece_rows == 8 && (pg0 + npg - 1) * 16 + 8 >= ctx;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], 2u * (npg * page_bytes - (tail_half ? page_bytes / 2 : 0u)));
      __syncwarp();
      // lanes < npg copy K pages, lanes npg..2npg-1 the V pages
      if (lane < 2 * npg) {
        const int which = lane >= npg ? 1 : 0;
        const int pg = lane - which * npg;
        const int tok = (pg0 + pg) * 16;
        bf16* dst = stages + static_cast<int64_t>(s) * 2 * C::kStageElems + which * C::kStageElems +
                    pg * page_elems;
        for (int r = 0; r < 16 && tok + r < ctx; r += piece_rows) {
          const int tr = tok + r;
          int blk = p.block_tables[static_cast<int64_t>(b) * p.bt_stride + (tr >> sh)];
          if (blk < 0 || blk >= p.num_blocks) {
            raise_error(p.err, PKV_DEVERR_BLOCK_RANGE);
            blk = 0;
          }
          const bf16* src = (which ? p.v_cache : p.k_cache) +
                            ((static_cast<int64_t>(blk) << sh) + (tr & bmask)) * row_elems;
          bulk_g2s(dst + r * row_elems, src, page_bytes / (16 / piece_rows), &full[s], pol);
        }
      }
    }
    // do not leave while this warp's copies may still be landing: the last fill of each
    // stage is the final phase of its full barrier, so waiting on it is safe (bounded)
    const int issued = it;
    for (int k = max(0, issued - STAGES); k < issued; ++k)
      wait_or_abort(&full[k % STAGES], (k / STAGES) & 1, p.err, abort_flag);
    return;
  }

  // -------------------------------------------------------------------- consumer warps
  const int pw = warp / hkv;  // page of the unit this warp reads
  const int h = warp - pw * hkv;  // kv head
  const int G_ = G;
  const float NEG_INF = -__int_as_float(0x7f800000);

  float qv[G][DPL], acc[G][DPL], m[G], lsum[G];
  int i = i_first;
  int ustart = 0, unext = 0, ctx = 0, npages = 0;
  int64_t tq = 0;
  bool seg_start = true;
  bool ok = true;
  int it = 0;
  for (int u = ubeg; u < uend; ++u, ++it) {
    if (seg_start) {
      if (i == i_first) {
        ustart = rec0.y;
        unext = rec0.z;
        ctx = rec1.x;
        tq = rec1.y;
      } else {
        ustart = dec_unit[i];
        unext = dec_unit[i + 1];
        ctx = p.plan.dec_ctx[i];
        tq = p.plan.dec_tq[i];
      }
      npages = ceil_div(ctx, 16);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const bf16* qrow = p.q + tq * p.q_st + static_cast<int64_t>(h * G_ + g) * p.q_sh;
        float x[DPL];
        load_row<DPL>(qrow, lane, true, x);
#pragma unroll
        for (int d = 0; d < DPL; ++d) {
          qv[g][d] = x[d] * p.qscale;
          acc[g][d] = 0.f;
        }
        m[g] = NEG_INF;
        lsum[g] = 0.f;
      }
      seg_start = false;
    }
    const int s = it % STAGES;
    if (ok) ok = wait_or_abort(&full[s], (it / STAGES) & 1, p.err, abort_flag);
    const int pg = (u - ustart) * pps + pw;
    if (ok && pg < npages) {
      const int rows = min(16, ctx - pg * 16);
      const bf16* Ks = stages + static_cast<int64_t>(s) * 2 * C::kStageElems + pw * page_elems + h * D;
      const bf16* Vs = Ks + C::kStageElems;
      const int rstride = hkv * D;

      // q . k partial sums over this lane's dims, 16 rows x G heads
      float part[16 * G];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float kf[DPL];
        load_row<DPL>(Ks + r * rstride, lane, r < rows, kf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float a = 0.f;
#pragma unroll
          for (int d = 0; d < DPL; ++d) a = fmaf(qv[g][d], kf[d], a);
          part[r * G + g] = a;
        }
      }
      // transposing butterfly: lane ends with the G full sums of row lane >> 1
      tr_level<8 * G>(part, 16, lane);
      tr_level<4 * G>(part, 8, lane);
      tr_level<2 * G>(part, 4, lane);
      tr_level<1 * G>(part, 2, lane);
#pragma unroll
      for (int g = 0; g < G; ++g) part[g] += __shfl_xor_sync(0xffffffffu, part[g], 1);

      const int row = lane >> 1;
      float pr[G];
      bool rescale = false;
      float corr[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float sc = row < rows ? part[g] : NEG_INF;
        float pm = sc;
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 2));
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
        const float mnew = fmaxf(m[g], pm);
        corr[g] = fast_exp2(m[g] - mnew);
        rescale |= (mnew != m[g]);
        m[g] = mnew;
        pr[g] = fast_exp2(sc - mnew);
        lsum[g] = lsum[g] * corr[g] + pr[g];
      }
      if (rescale) {  // warp-uniform: m is identical in every lane
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int d = 0; d < DPL; ++d) acc[g][d] *= corr[g];
      }
      float* pb = pbuf + warp * 16 * G;
      if ((lane & 1) == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) pb[row * G + g] = pr[g];
      }
      __syncwarp();
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        if (r < rows) {
          float vf[DPL];
          load_row<DPL>(Vs + r * rstride, lane, true, vf);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float w = pb[r * G + g];
#pragma unroll
            for (int d = 0; d < DPL; ++d) acc[g][d] = fmaf(w, vf[d], acc[g][d]);
          }
        }
      }
      __syncwarp();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    const bool seg_end = (u + 1 == unext) || (u + 1 == uend);
    if (!seg_end) continue;

    // ---------------------------------------------------------------- segment flush
    float L[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float x = lsum[g];
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      x += __shfl_xor_sync(0xffffffffu, x, 4);
      x += __shfl_xor_sync(0xffffffffu, x, 8);
      x += __shfl_xor_sync(0xffffffffu, x, 16);
      L[g] = x;
    }
    if (pps > 1) {
      if (warp >= hkv) {
        float* xb = xbuf + (warp - hkv) * G * (D + 2);
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
          for (int d = 0; d < DPL; ++d) xb[g * (D + 2) + lane * DPL + d] = acc[g][d];
          if (lane == 0) {
            xb[g * (D + 2) + D] = m[g];
            xb[g * (D + 2) + D + 1] = L[g];
          }
        }
      }
      named_bar_sync(1, kDecodeWarps * 32);
      if (warp < hkv) {
        for (int k = 1; k < pps; ++k) {
          const float* xb = xbuf + (warp + k * hkv - hkv) * G * (D + 2);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float mo = xb[g * (D + 2) + D];
            const float lo = xb[g * (D + 2) + D + 1];
            const float mn = fmaxf(m[g], mo);
            const float fa = fast_exp2(m[g] - mn);
            const float fb = fast_exp2(mo - mn);
            L[g] = L[g] * fa + lo * fb;
#pragma unroll
            for (int d = 0; d < DPL; ++d)
              acc[g][d] = acc[g][d] * fa + xb[g * (D + 2) + lane * DPL + d] * fb;
            m[g] = mn;
          }
        }
      }
      named_bar_sync(1, kDecodeWarps * 32);
    }
    if (warp < hkv) {
      const int chunks = p.plan.dec_chunks[i];
      if (chunks == 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float inv = 1.f / L[g];
          bf16* orow = p.out + tq * p.o_st + static_cast<int64_t>(h * G_ + g) * p.o_sh + lane * DPL;
          if constexpr (DPL == 4) {
            uint2 w;
            w.x = pack_bf16x2(acc[g][0] * inv, acc[g][1] * inv);
            w.y = pack_bf16x2(acc[g][2] * inv, acc[g][3] * inv);
            *reinterpret_cast<uint2*>(orow) = w;
          } else {
            *reinterpret_cast<uint32_t*>(orow) = pack_bf16x2(acc[g][0] * inv, acc[g][1] * inv);
          }
        }
      } else {
        const int slot = p.plan.dec_slot[i] + (static_cast<int>(blockIdx.x) - ustart / W);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int hq = h * G_ + g;
          float* pa = p.plan.part_acc + (static_cast<int64_t>(slot) * p.hq + hq) * D + lane * DPL;
          if constexpr (DPL == 4) {
            *reinterpret_cast<float4*>(pa) = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
          } else {
            *reinterpret_cast<float2*>(pa) = make_float2(acc[g][0], acc[g][1]);
          }
          if (lane == 0)
            *reinterpret_cast<float2*>(p.plan.part_ml + (static_cast<int64_t>(slot) * p.hq + hq) * 2) =
                make_float2(m[g], L[g]);
        }
      }
    }
    if (p.plan.dec_chunks[i] > 1) finish_split<D>(p, i, tq, p.plan.dec_chunks[i], p.plan.dec_slot[i], last_flag);
    seg_start = true;
    ++i;
  }
}

}  // namespace pkv
