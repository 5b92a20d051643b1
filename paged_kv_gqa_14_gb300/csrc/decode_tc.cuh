// Decode split-K on the tensor cores: the GQA group is the contraction's N dimension.
//
// Same work decomposition, producer/consumer ring and split states as the CUDA-core
// decode kernel (decode.cuh): a unit is P = 8 / Hkv pages of one decode sequence with all kv
// heads, consumer warp w owns page w / Hkv and kv head w % Hkv, and every K/V page is read
// from HBM once per GQA group.  What changes is the arithmetic of a (page, kv head):
//
//   S^T [16 tokens x 8] = K_page [16 x d] . Q_g^T [d x 8]       mma.sync m16n8k16, bf16 -> fp32
//   online softmax over the 16 token rows of each head column (warp shuffles)
//   P^T packed to bf16 and transposed in registers with movmatrix
//   O^T [d x 8]        += V_page^T [d x 16] . P^T [16 x 8]       mma.sync m16n8k16
//
// M = the page's 16 tokens, N = 8 >= G query heads (unused columns are zero q), K = d for
// QK^T and 16 tokens for PV.  This removes the G-proportional CUDA-core work (G FMAs per
// loaded element plus shuffle reductions) that caps the scalar kernel at large G.
//
// K/V pages are staged by 4-D TMA tensor loads over the pool viewed head-major,
// {d, block rows, Hkv, num_blocks} (strides: a row, a head, a block): one box is 64 dims x
// 16 token rows x all kv heads of a page, landing as [kv head][16 rows][128 bytes] with the
// 128-byte swizzle, so the ldmatrix reads of 8 token rows of one head hit 8 different bank
// groups.  One box per (page, 64-dim half) instead of one per kv head: on GB300 per-head
// boxes of 2 KB moved 4.6 TB/s from HBM in a copy-only test, page-wide boxes 6.1 TB/s.  A
// 16-token page is rows 16j..16j+15 of one block when blocks hold 16 or more tokens; with
// 8-token blocks it is two boxes of 8 rows from two blocks, [row half][kv head][8 rows].
//
// The producer requests a unit's block ids before it waits for the unit's stage, and with
// early streaming it starts on the plan's ready word instead of the planner's end, waiting for
// the kernel before the planner only before the first page that may hold a new key; the
// consumers wait for it before they read q.
//
// The kernel is instantiated per block size, with it folded in at compile time.  The decode
// is sensitive to the producer warp's instruction stream (the warp shares a scheduler with
// two consumer warps and sits on the ring's refill path): on GB300 a form reading the block
// size at run time cost about 8% of decode time at 16-token blocks.  The instances live in
// decode_tc.cu, built once per block size.
#pragma once

#include <cuda.h>

#include "decode.cuh"

namespace pkv {

struct DecodeTcParams {
  CUtensorMap tmap_k;  // 4-D: {d, block_size, Hkv, num_blocks}, box {64, min(block_size, 16), Hkv, 1}, 128B swizzle
  CUtensorMap tmap_v;
  DecodeParams p;
};

template <int D, int G>
struct DecodeTcCfg {
  static constexpr int HALVES = D / 64;                 // 64-dim boxes per head row
  static constexpr int kBoxBytes = 16 * 64 * 2;         // one box: 16 tokens x 64 dims
  static constexpr int kPartBytes = kDecodeWarps * HALVES * kBoxBytes;  // K (or V) of a stage
  static constexpr int kStageBytes = 2 * kPartBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kXbufBytes = kDecodeWarps * G * (D + 2) * 4;
  static constexpr int kReserve = kBarBytes + kXbufBytes + 1024;  // + alignment slack
  static constexpr int kSmemLimit = 227 * 1024;
  static constexpr int kStagesFit = (kSmemLimit - kReserve) / kStageBytes;
  static constexpr int STAGES = kStagesFit > 4 ? 4 : kStagesFit;
  static constexpr int kSmemBytes = STAGES * kStageBytes + kReserve;
  static_assert(STAGES >= 2, "decode pipeline needs at least two stages");
  static_assert(G >= 1 && G <= 8, "the GQA group is the mma N dimension (8)");
};

__device__ __forceinline__ void tma_load_4d(void* dst_smem, const CUtensorMap* map, int c0, int c1, int c2,
                                            int c3, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst_smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4_tc(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t_tc(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// byte offset of 16-byte chunk `c` (0..7) of token row `t` inside its 8-row, 1024-byte
// 128B-swizzled atom (rows t and t + 8 sit in two atoms)
__device__ __forceinline__ uint32_t chunk_off(int t, int c) { return (t & 7) * 128 + ((c ^ (t & 7)) << 4); }

// BS: tokens per pool block, a power of two from 8 to 128.
template <int D, int G, int BS>
__global__ void __launch_bounds__((kDecodeWarps + 1) * 32, 1)
    decode_tc_kernel(const __grid_constant__ DecodeTcParams P) {
  using C = DecodeTcCfg<D, G>;
  constexpr int STAGES = C::STAGES;
  constexpr int HALVES = C::HALVES;
  constexpr int KS = D / 16;  // k-steps of QK^T, m-tiles of PV
  const DecodeParams& p = P.p;
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte alignment for the 128B swizzle pattern
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
  uint64_t* empty = full + STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STAGES);
  volatile int* last_flag = abort_flag + 2;
  volatile int* stream_mode = abort_flag + 4;
  float* xbuf = reinterpret_cast<float*>(smem + STAGES * C::kStageBytes + C::kBarBytes);

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
  if (warp == kDecodeWarps && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_v)) : "memory");
  }
  // The plan is written by the planner kernel.  Streaming early, the CTA reads it as soon as
  // the planner has published it (mode 1 or 2, see the ready word); the producer then copies
  // pages while the kernel before the planner may still run, and waits for that kernel only
  // before the first page that may hold a new key (mode 1: an entry's last page; mode 2: any),
  // and the consumers before they read q.  Mode 0: everything before this kernel has finished.
  int mode = 0;
  if (p.stream_early) {
    if (threadIdx.x == 0) {
      int v;
      const long long t0 = clock64();
      while ((v = ld_acquire_gpu(p.plan.header + kPlanReadyWord)) == 0 && clock64() - t0 < kPlanReadySpinClocks)
        __nanosleep(64);
      *stream_mode = v;  // still 0 at the limit: every thread waits for the planner's end instead
    }
    __syncthreads();
    mode = *stream_mode;
    if (mode == 0) pdl_wait();
  } else {
    pdl_wait();
  }
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
  const uint32_t page_bytes = static_cast<uint32_t>(hkv * HALVES * C::kBoxBytes);
  // shared-memory image of a stage: [K|V][page][64-dim half][kv head][16 rows][128 B]; with
  // 8-token blocks [K|V][page][half][row half][kv head][8 rows][128 B]
  const uint32_t hstride = static_cast<uint32_t>(hkv * C::kBoxBytes);  // one (page, half) of all heads
  constexpr bool two_block_pages = BS == 8;
  const uint32_t head_off = two_block_pages ? 1024u : static_cast<uint32_t>(C::kBoxBytes);  // next kv head
  const uint32_t rowhalf_off = two_block_pages ? static_cast<uint32_t>(hkv * 1024) : 1024u;  // rows 8..15

  if (warp == kDecodeWarps) {
    // ------------------------------------------------------------------ producer warp
    // Fault injection for the tests of the bounded waits: no copy and no arrival is issued,
    // so the consumers' first waits run out, set PKV_DEVERR_TIMEOUT and the CTA finishes.
    if (p.fault_no_copies) return;
    const uint64_t pol = l2_policy_evict_first();
    // lane -> (K or V, page, 64-dim half) of the unit's boxes; 2 P HALVES <= 32 boxes
    const int per_kv = pps * HALVES;
    const int kv = lane / per_kv;
    const int rem = lane - kv * per_kv;
    const int bp = rem / HALVES;
    const int bhalf = rem - bp * HALVES;
    const bool lane_has_box = lane < 2 * per_kv;
    int i = i_first;
    int ustart = rec0.y, unext = rec0.z;
    int b = rec0.w;
    int ctx = rec1.x;
    int npages = ceil_div(ctx, 16);
    // page gp: block gp >> s4 and its rows from (16 gp) & bmask when blocks hold 16 << s4
    // tokens; blocks 2 gp and 2 gp + 1 (the second only if it holds context) when they hold 8
    constexpr int sh = BS == 8 ? 3 : BS == 16 ? 4 : BS == 32 ? 5 : BS == 64 ? 6 : 7;
    static_assert((1 << sh) == BS, "block size must be a power of two from 8 to 128");
    constexpr int bmask = BS - 1;
    constexpr bool two_blocks = BS == 8;
    int it = 0;
    bool waited = mode == 0;
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
      int blk = 0, blk2 = -1;
      const bool issue = lane_has_box && bp < npg;
      const int gp = pg0 + bp;
      if (issue) {
        // the unit's block ids are requested before the wait for its stage, so their latency
        // passes while the ring is full, and a freed stage is refilled at once; both reads are
        // issued before either is checked
        const int32_t* row = p.block_tables + static_cast<int64_t>(b) * p.bt_stride;
        blk = row[two_blocks ? 2 * gp : gp >> (sh >= 4 ? sh - 4 : 0)];
        if (two_blocks && gp * 16 + 8 < ctx) blk2 = row[2 * gp + 1];
      }
      if (it >= STAGES && !wait_or_abort(&empty[s], ((it / STAGES) - 1) & 1, p.err, abort_flag)) break;
      if (issue) {
        if (blk < 0 || blk >= p.num_blocks) {
          raise_error(p.err, PKV_DEVERR_BLOCK_RANGE);
          blk = 0;
        }
        if (two_blocks && gp * 16 + 8 < ctx && (blk2 < 0 || blk2 >= p.num_blocks)) {
          raise_error(p.err, PKV_DEVERR_BLOCK_RANGE);
          blk2 = 0;
        }
      }
      if (!waited && (mode == 2 || pg0 + npg - 1 >= (ctx - 1) >> 4)) {
        pdl_wait();  // this unit may hold a key written by the kernel before the planner
        waited = true;
      }
      // a last half page past the context is not loaded (8-token blocks)
      const bool tail_half = two_blocks && (pg0 + npg - 1) * 16 + 8 >= ctx;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], 2u * (npg * page_bytes - (tail_half ? page_bytes / 2 : 0u)));
      __syncwarp();
      if (issue) {
        unsigned char* dst = stages + s * C::kStageBytes + kv * C::kPartBytes + (bp * HALVES + bhalf) * hstride;
        const CUtensorMap* map = kv ? &P.tmap_v : &P.tmap_k;
        tma_load_4d(dst, map, bhalf * 64, (gp * 16) & bmask, 0, blk, &full[s], pol);
        if (blk2 >= 0) tma_load_4d(dst + hkv * 1024, map, bhalf * 64, 0, 0, blk2, &full[s], pol);
      }
    }
    const int issued = it;
    for (int k = max(0, issued - STAGES); k < issued; ++k)
      wait_or_abort(&full[k % STAGES], (k / STAGES) & 1, p.err, abort_flag);
    return;
  }

  // -------------------------------------------------------------------- consumer warps
  if (mode != 0) pdl_wait();  // q is written by the kernel before the planner
  const int pw = warp / hkv;
  const int h = warp - pw * hkv;
  const int gr = lane >> 2, tig = lane & 3;
  const float NEG_INF = -__int_as_float(0x7f800000);

  uint32_t qb[KS][2];  // Q^T B fragments: head gr (zero past G), dims of k-step kk
  float acc[KS][4];    // O^T: dims 16mt + gr (+8), heads 2tig (+1)
  float mrun[2], lrun[2];
  int i = i_first;
  int ustart = 0, unext = 0, ctx = 0, npages = 0;
  int64_t tq = 0;
  bool seg_start = true;
  bool ok = true;
  int it = 0;
  const uint32_t stage_base = smem_u32(stages);
  const bool hv = gr < G;
  // The next segment's entry (i + 1), when it starts inside this CTA's range, is read while
  // this segment runs: its unit end, context and query row at this segment's start, its Q
  // fragments after this segment's first unit.  A segment boundary then waits on no global
  // read, while the producer's ring stays full.
  int nx_unext = 0, nx_ctx = 0;
  int64_t nx_tq = 0;
  uint32_t nx_qb[KS][2];
  bool nx_pending = false, nx_have_q = false;
  int chunks = 1, slot0 = 0;  // the current entry's split pieces and first split slot
  auto load_q = [&](int64_t row_tq, uint32_t (&dst)[KS][2]) {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        p.q + row_tq * p.q_st + static_cast<int64_t>(h * G + (hv ? gr : 0)) * p.q_sh);
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      dst[kk][0] = hv ? qrow[kk * 8 + tig] : 0u;
      dst[kk][1] = hv ? qrow[kk * 8 + 4 + tig] : 0u;
    }
  };
  for (int u = ubeg; u < uend; ++u, ++it) {
    if (seg_start) {
      if (i == i_first) {
        ustart = rec0.y;
        unext = rec0.z;
        ctx = rec1.x;
        tq = rec1.y;
        load_q(tq, qb);
      } else {
        ustart = unext;  // entries are consecutive: this one starts where the last one ended
        unext = nx_unext;
        ctx = nx_ctx;
        tq = nx_tq;
        if (nx_have_q) {
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            qb[kk][0] = nx_qb[kk][0];
            qb[kk][1] = nx_qb[kk][1];
          }
        } else {
          load_q(tq, qb);
        }
      }
      npages = ceil_div(ctx, 16);
      chunks = p.plan.dec_chunks[i];
      slot0 = p.plan.dec_slot[i];
      nx_pending = unext < uend;
      nx_have_q = false;
      if (nx_pending) {
        nx_unext = dec_unit[i + 2];
        nx_ctx = p.plan.dec_ctx[i + 1];
        nx_tq = p.plan.dec_tq[i + 1];
      }
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
      mrun[0] = mrun[1] = NEG_INF;
      lrun[0] = lrun[1] = 0.f;
      seg_start = false;
    }
    const int s = it % STAGES;
    if (ok) ok = wait_or_abort(&full[s], (it / STAGES) & 1, p.err, abort_flag);
    const int pg = (u - ustart) * pps + pw;
    if (ok && pg < npages) {
      const int rows = min(16, ctx - pg * 16);
      const uint32_t kbox = stage_base + s * C::kStageBytes + pw * HALVES * hstride + h * head_off;
      const uint32_t vbox = kbox + C::kPartBytes;
      if (rows < 16) {
        // keys past the context: zero their V rows so 0 * (unused slot) cannot poison P.V
        unsigned char* vgen = stages + s * C::kStageBytes + C::kPartBytes + pw * HALVES * hstride + h * head_off;
        for (int idx = lane; idx < (16 - rows) * 8 * HALVES; idx += 32) {
          const int hh = idx / ((16 - rows) * 8);
          const int r2 = idx - hh * (16 - rows) * 8;
          const int t = rows + (r2 >> 3);
          *reinterpret_cast<uint4*>(vgen + hh * hstride + (t >> 3) * rowhalf_off + (t & 7) * 128 + ((r2 & 7) << 4)) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      // S^T = K . Q^T
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int r = (lane & 7) + 8 * ((lane >> 3) & 1);
        const uint32_t rsel = (r >> 3) * rowhalf_off;
        const int csel = lane >> 4;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          uint32_t a[4];
          ldsm_x4_tc(a, kbox + (kk >> 2) * hstride + rsel + chunk_off(r, 2 * (kk & 3) + csel));
          mma_16816(sc, a, qb[kk][0], qb[kk][1]);
        }
      }
      // scale, mask, online softmax over the token rows of each head column
      const bool v0 = gr < rows, v1 = gr + 8 < rows;
      sc[0] = v0 ? sc[0] * p.qscale : NEG_INF;
      sc[1] = v0 ? sc[1] * p.qscale : NEG_INF;
      sc[2] = v1 ? sc[2] * p.qscale : NEG_INF;
      sc[3] = v1 ? sc[3] * p.qscale : NEG_INF;
      float pm0 = fmaxf(sc[0], sc[2]), pm1 = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        pm0 = fmaxf(pm0, __shfl_xor_sync(0xffffffffu, pm0, off));
        pm1 = fmaxf(pm1, __shfl_xor_sync(0xffffffffu, pm1, off));
      }
      const float mn0 = fmaxf(mrun[0], pm0), mn1 = fmaxf(mrun[1], pm1);
      const float c0 = fast_exp2(mrun[0] - mn0), c1 = fast_exp2(mrun[1] - mn1);
      mrun[0] = mn0;
      mrun[1] = mn1;
      sc[0] = fast_exp2(sc[0] - mn0);
      sc[1] = fast_exp2(sc[1] - mn1);
      sc[2] = fast_exp2(sc[2] - mn0);
      sc[3] = fast_exp2(sc[3] - mn1);
      lrun[0] = lrun[0] * c0 + sc[0] + sc[2];
      lrun[1] = lrun[1] * c1 + sc[1] + sc[3];
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        acc[mt][0] *= c0;
        acc[mt][1] *= c1;
        acc[mt][2] *= c0;
        acc[mt][3] *= c1;
      }
      // P^T (tokens x heads) -> B fragments (k = token, n = head) by an 8x8 transpose
      const uint32_t pb0 = movmatrix_t(pack_bf16x2(sc[0], sc[1]));
      const uint32_t pb1 = movmatrix_t(pack_bf16x2(sc[2], sc[3]));
      // O^T += V^T . P^T
      {
        const int r = (lane & 7) + 8 * (lane >> 4);
        const uint32_t rsel = (r >> 3) * rowhalf_off;
        const int csel = (lane >> 3) & 1;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          uint32_t a[4];
          ldsm_x4_t_tc(a, vbox + (mt >> 2) * hstride + rsel + chunk_off(r, 2 * (mt & 3) + csel));
          mma_16816(acc[mt], a, pb0, pb1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (nx_pending && !nx_have_q) {  // (the next entry's query row has arrived by now)
      load_q(nx_tq, nx_qb);
      nx_have_q = true;
    }

    const bool seg_end = (u + 1 == unext) || (u + 1 == uend);
    if (!seg_end) continue;

    // ---------------------------------------------------------------- segment flush
    float L0 = lrun[0], L1 = lrun[1];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      L0 += __shfl_xor_sync(0xffffffffu, L0, off);
      L1 += __shfl_xor_sync(0xffffffffu, L1, off);
    }
    float* xb = xbuf + warp * G * (D + 2);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int hh = 2 * tig + j;
      if (hh < G) {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          xb[hh * (D + 2) + 16 * mt + gr] = acc[mt][j];
          xb[hh * (D + 2) + 16 * mt + gr + 8] = acc[mt][2 + j];
        }
        if (gr == 0) {
          xb[hh * (D + 2) + D] = mrun[j];
          xb[hh * (D + 2) + D + 1] = j ? L1 : L0;
        }
      }
    }
    named_bar_sync(1, kDecodeWarps * 32);
    {
      const int slot = slot0 + (static_cast<int>(blockIdx.x) - ustart / W);
      const int tid = threadIdx.x;  // 0..255
      for (int item = tid; item < hkv * G * (D / 4); item += kDecodeWarps * 32) {
        const int hh = item / (G * (D / 4));
        const int rem3 = item - hh * G * (D / 4);
        const int g = rem3 / (D / 4);
        const int d0 = (rem3 - g * (D / 4)) * 4;
        float M = NEG_INF;
        for (int k = 0; k < pps; ++k) M = fmaxf(M, xbuf[((hh + k * hkv) * G + g) * (D + 2) + D]);
        float num[4] = {0.f, 0.f, 0.f, 0.f};
        float den = 0.f;
        for (int k = 0; k < pps; ++k) {
          const float* e = xbuf + ((hh + k * hkv) * G + g) * (D + 2);
          const float w = fast_exp2(e[D] - M);  // a warp with no pages: m = -inf -> w = 0
          den = fmaf(w, e[D + 1], den);
#pragma unroll
          for (int x = 0; x < 4; ++x) num[x] = fmaf(w, e[d0 + x], num[x]);
        }
        const int hq = hh * G + g;
        if (chunks == 1) {
          const float inv = 1.f / den;
          uint2 o;
          o.x = pack_bf16x2(num[0] * inv, num[1] * inv);
          o.y = pack_bf16x2(num[2] * inv, num[3] * inv);
          *reinterpret_cast<uint2*>(p.out + tq * p.o_st + static_cast<int64_t>(hq) * p.o_sh + d0) = o;
        } else {
          const int64_t sh = static_cast<int64_t>(slot) * p.hq + hq;
          *reinterpret_cast<float4*>(p.plan.part_acc + sh * D + d0) = make_float4(num[0], num[1], num[2], num[3]);
          if (d0 == 0) *reinterpret_cast<float2*>(p.plan.part_ml + sh * 2) = make_float2(M, den);
        }
      }
    }
    named_bar_sync(1, kDecodeWarps * 32);
    if (chunks > 1) finish_split<D>(p, i, tq, chunks, slot0, last_flag);
    seg_start = true;
    ++i;
  }
}

// The pool [num_blocks][block_size][Hkv][d] as a 4-D tensor map for the tensor-core
// kernels (defined in attention.cu).
bool make_pool_map(CUtensorMap* m, const void* base, int64_t num_blocks, int bs_log2, int hkv, int D);
// The same pool viewed head-major (page-wide boxes of all kv heads), for the decode.
bool make_pool_map_heads(CUtensorMap* m, const void* base, int64_t num_blocks, int bs_log2, int hkv, int D);

}  // namespace pkv
