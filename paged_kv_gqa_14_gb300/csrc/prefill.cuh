// Prefill-chunk kernel: causal attention of a span of n > 1 new tokens over its whole paged
// context ("mini_engine" README, "What it does": chunked prefill under
// max_num_batched_tokens; "09 -- Mini Inference Engine (The Capstone)", "Week 3": mixed
// prefill/decode batches of varying lengths).
//
// Work item: (sequence, 64-row q tile of its span, q head).  Row r of an n-row span sits at
// position ctx - n + r and sees keys 0 .. ctx - n + r.  Four warps each own 16 q rows.
// K/V tiles of 64 keys (four 16-token pages, gathered through the block table) are staged
// with cp.async into XOR-swizzled shared memory, double buffered; QK^T and PV run on the
// tensor cores as bf16 mma.sync m16n8k16 with fp32 accumulation, the probabilities staying
// in registers between the two products.  Keys past the context are zero-filled, masked
// scores are selected to -inf (never multiplied), so NaN in unused pool slots cannot leak.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace pkv {

struct PrefillParams {
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
};

// Persistent grids walk the work list heaviest first (the planner lists each span's tiles in
// order, later tiles see more keys) in a snake: even waves left to right, odd waves right to
// left, so the CTA that took the heaviest item of one wave takes the lightest of the next.
__device__ __forceinline__ int snake_order(int wave, int cta, int ctas) {
  return wave * ctas + ((wave & 1) ? ctas - 1 - cta : cta);
}

template <int D>
struct PrefillCfg {
  static constexpr int TQ = kPrefillTileQ;  // q rows per work item
  static constexpr int TK = 64;             // keys per K/V tile
  static constexpr int CH = D / 8;          // 16-byte chunks per row
  static constexpr int kTileElems = 64 * D;
  static constexpr int kThreads = 128;
  static constexpr int kSmemBytes = 5 * kTileElems * 2;  // Q + 2 x K + 2 x V
  static_assert(TQ == 64 && TK == 64, "tile shape");
};

// position (in 16-byte chunks) of chunk `c` of row `r` in a swizzled tile
template <int CH>
__device__ __forceinline__ int swz(int r, int c) {
  return r * CH + (c ^ (r & 7));
}

__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes: zero fill
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst_smem)), "l"(src),
               "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2_pf(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
__device__ __forceinline__ void load_kv_tile(bf16* sK, bf16* sV, const PrefillParams& p, int b, int h,
                                             int kt, int kv_end) {
  using C = PrefillCfg<D>;
  const int64_t row_elems = static_cast<int64_t>(p.hkv) * D;
  for (int c = threadIdx.x; c < 64 * C::CH; c += C::kThreads) {
    const int r = c / C::CH;
    const int ch = c - r * C::CH;
    const int key = kt * 64 + r;
    const bool valid = key < kv_end;
    int blk = 0;
    if (valid) {
      blk = p.block_tables[static_cast<int64_t>(b) * p.bt_stride + (key >> p.bs_log2)];
      if (blk < 0 || blk >= p.num_blocks) {
        raise_error(p.err, PKV_DEVERR_BLOCK_RANGE);
        blk = 0;
      }
    }
    const int64_t off =
        ((static_cast<int64_t>(blk) << p.bs_log2) + (key & ((1 << p.bs_log2) - 1))) * row_elems + h * D + ch * 8;
    cp_async16(sK + swz<C::CH>(r, ch) * 8, p.k_cache + (valid ? off : 0), valid);
    cp_async16(sV + swz<C::CH>(r, ch) * 8, p.v_cache + (valid ? off : 0), valid);
  }
}

template <int D>
__global__ void __launch_bounds__(128) prefill_kernel(const __grid_constant__ PrefillParams p) {
  using C = PrefillCfg<D>;
  constexpr int KS = D / 16;  // k-steps over head_dim
  constexpr int NT = D / 8;   // 8-wide output tiles over head_dim
  extern __shared__ __align__(128) unsigned char smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sK = sQ + C::kTileElems;
  bf16* sV = sK + 2 * C::kTileElems;
  const float NEG_INF = -__int_as_float(0x7f800000);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, tig = lane & 3;
  pdl_wait();  // the tile list is written by the planner kernel (on a second stream an event orders it)
  pdl_trigger();
  const int n_tiles = p.plan.header[3];
  const int total = n_tiles * p.hq;
  const int G = p.hq / p.hkv;
  // the planner's count of CTAs that take items (fewer than launched when the prefill
  // shares the SMs with the decode); the others leave
  const int nact = min(max(p.plan.header[5], 0), static_cast<int>(gridDim.x));
  if (static_cast<int>(blockIdx.x) >= nact) return;

  for (int wave = 0; wave * nact < total; ++wave) {
    const int ord = snake_order(wave, blockIdx.x, nact);
    if (ord >= total) continue;
    const int item = total - 1 - ord;  // later (longer) tiles of each span first
    const int ti = item / p.hq;
    const int hq = item - ti * p.hq;
    const int h = hq / G;
    const int b = p.plan.pf_seq[ti];
    const int j = p.plan.pf_tile[ti];
    const int s0 = p.qsl[b];
    const int n = p.qsl[b + 1] - s0;
    const int ctx = p.context_lens[b];
    const int q0 = j * C::TQ;
    const int qrows = min(C::TQ, n - q0);
    const int pos0 = ctx - n + q0;       // position of the tile's first row
    const int kv_end = pos0 + qrows;     // keys [0, kv_end) are visible to some row
    const int nkt = ceil_div(kv_end, C::TK);

    // Q tile (rows past the span are zero) and the first K/V tile
    for (int c = threadIdx.x; c < 64 * C::CH; c += C::kThreads) {
      const int r = c / C::CH;
      const int ch = c - r * C::CH;
      const bool valid = r < qrows;
      const bf16* src = p.q + (valid ? (static_cast<int64_t>(s0 + q0 + r) * p.q_st + hq * p.q_sh + ch * 8) : 0);
      cp_async16(sQ + swz<C::CH>(r, ch) * 8, src, valid);
    }
    load_kv_tile<D>(sK, sV, p, b, h, 0, kv_end);
    cp_async_commit();

    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mrow[2] = {NEG_INF, NEG_INF};
    float lrow[2] = {0.f, 0.f};
    uint32_t qa[KS][4];
    const int rbase = warp * 16;  // this warp's first row in the tile
    const int pos_r0 = pos0 + rbase + gr;  // positions of the lane's two rows
    const int pos_r1 = pos_r0 + 8;
    const bool live0 = rbase + gr < qrows, live1 = rbase + gr + 8 < qrows;

    for (int kt = 0; kt < nkt; ++kt) {
      const int buf = kt & 1;
      if (kt + 1 < nkt) {
        load_kv_tile<D>(sK + (buf ^ 1) * C::kTileElems, sV + (buf ^ 1) * C::kTileElems, p, b, h, kt + 1, kv_end);
        cp_async_commit();
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      if (kt == 0) {
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int r = rbase + (lane & 7) + 8 * ((lane >> 3) & 1);
          ldsm_x4(qa[kk], sQ + swz<C::CH>(r, 2 * kk + (lane >> 4)) * 8);
        }
      }
      const bf16* tK = sK + buf * C::kTileElems;
      const bf16* tV = sV + buf * C::kTileElems;

      // S = Q K^T for this warp's 16 rows x 64 keys
      float s[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t bfr[4];
          const int kr = np * 16 + (lane & 7) + 8 * (lane >> 4);
          ldsm_x4(bfr, tK + swz<C::CH>(kr, 2 * kk + ((lane >> 3) & 1)) * 8);
          mma_bf16(s[2 * np], qa[kk], bfr[0], bfr[1]);
          mma_bf16(s[2 * np + 1], qa[kk], bfr[2], bfr[3]);
        }
      }
      // scale, causal mask (select, NaN-safe), online softmax in the log2 domain
      float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int key = kt * 64 + nt * 8 + tig * 2;
        s[nt][0] = (live0 && key <= pos_r0) ? s[nt][0] * p.qscale : NEG_INF;
        s[nt][1] = (live0 && key + 1 <= pos_r0) ? s[nt][1] * p.qscale : NEG_INF;
        s[nt][2] = (live1 && key <= pos_r1) ? s[nt][2] * p.qscale : NEG_INF;
        s[nt][3] = (live1 && key + 1 <= pos_r1) ? s[nt][3] * p.qscale : NEG_INF;
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(mrow[0], mx0), mn1 = fmaxf(mrow[1], mx1);
      const float base0 = mn0 == NEG_INF ? 0.f : mn0;  // all masked so far: keep weights 0
      const float base1 = mn1 == NEG_INF ? 0.f : mn1;
      const float c0 = fast_exp2_pf(mrow[0] - base0), c1 = fast_exp2_pf(mrow[1] - base1);
      mrow[0] = mn0;
      mrow[1] = mn1;
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        s[nt][0] = fast_exp2_pf(s[nt][0] - base0);
        s[nt][1] = fast_exp2_pf(s[nt][1] - base0);
        s[nt][2] = fast_exp2_pf(s[nt][2] - base1);
        s[nt][3] = fast_exp2_pf(s[nt][3] - base1);
        ls0 += s[nt][0] + s[nt][1];
        ls1 += s[nt][2] + s[nt][3];
      }
      lrow[0] = lrow[0] * c0 + ls0;
      lrow[1] = lrow[1] * c1 + ls1;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        o[i][0] *= c0;
        o[i][1] *= c0;
        o[i][2] *= c1;
        o[i][3] *= c1;
      }
      // O += P V
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t pa[4];
        pa[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
        pa[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
        pa[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        pa[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          uint32_t bfr[4];
          const int kr = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
          ldsm_x4_t(bfr, tV + swz<C::CH>(kr, 2 * dp + (lane >> 4)) * 8);
          mma_bf16(o[2 * dp], pa, bfr[0], bfr[1]);
          mma_bf16(o[2 * dp + 1], pa, bfr[2], bfr[3]);
        }
      }
      __syncthreads();  // this buffer is refilled two iterations from now
    }

    // normalise and write the live rows
    lrow[0] += __shfl_xor_sync(0xffffffffu, lrow[0], 1);
    lrow[0] += __shfl_xor_sync(0xffffffffu, lrow[0], 2);
    lrow[1] += __shfl_xor_sync(0xffffffffu, lrow[1], 1);
    lrow[1] += __shfl_xor_sync(0xffffffffu, lrow[1], 2);
    const float inv0 = live0 ? 1.f / lrow[0] : 0.f;
    const float inv1 = live1 ? 1.f / lrow[1] : 0.f;
    bf16* orow0 = p.out + static_cast<int64_t>(s0 + q0 + rbase + gr) * p.o_st + hq * p.o_sh;
    bf16* orow1 = orow0 + 8 * p.o_st;
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int d = i * 8 + tig * 2;
      if (live0) *reinterpret_cast<uint32_t*>(orow0 + d) = pack_bf16x2(o[i][0] * inv0, o[i][1] * inv0);
      if (live1) *reinterpret_cast<uint32_t*>(orow1 + d) = pack_bf16x2(o[i][2] * inv1, o[i][3] * inv1);
    }
  }
}

inline PrefillParams make_prefill_params(const AttnArgs& a) {
  PrefillParams p;
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
  return p;
}

// CTAs the mma.sync prefill is launched with: two per SM, at most one per item.
inline int64_t prefill_mma_grid(const AttnArgs& a) {
  const int64_t max_items = a.max_tiles * a.hq;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 2;
  return max_items < cap ? max_items : cap;
}

template <int D>
cudaError_t launch_prefill(const AttnArgs& a, cudaStream_t stream, bool pdl) {
  using C = PrefillCfg<D>;
  if (const cudaError_t e = set_smem_once<prefill_kernel<D>>(C::kSmemBytes); e != cudaSuccess) return e;
  const PrefillParams p = make_prefill_params(a);
  const unsigned grid = static_cast<unsigned>(prefill_mma_grid(a));
  if (grid == 0) return cudaSuccess;
  record_kernel_event(PKV_KERNEL_PREFILL, false, stream);
  const cudaError_t e =
      launch_kernel(pdl, prefill_kernel<D>, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream, p);
  record_kernel_event(PKV_KERNEL_PREFILL, true, stream);
  return e;
}

}  // namespace pkv
