// Launchers of the tensor-core decode kernel (decode_tc.cuh) for one pool block size.
//
// This file is compiled once per supported block size with -DPKV_DECODE_TC_BS=<size>; each
// object defines launch_decode_tc_bs<size>() covering every head dim and GQA group.  Keeping
// the block size a compile-time constant keeps the producer warp's page walk as short as
// the 16-token case's, and one translation unit per size lets the build compile them in
// parallel.
#include "decode_tc.cuh"

#ifndef PKV_DECODE_TC_BS
#error "compile with -DPKV_DECODE_TC_BS=<block size>"
#endif

#define PKV_CAT2(a, b) a##b
#define PKV_CAT(a, b) PKV_CAT2(a, b)

namespace pkv {
namespace {

constexpr int BS = PKV_DECODE_TC_BS;

template <int D, int G>
cudaError_t launch(const AttnArgs& a, cudaStream_t stream) {
  using C = DecodeTcCfg<D, G>;
  if (const cudaError_t e = set_smem_once<decode_tc_kernel<D, G, BS>>(C::kSmemBytes); e != cudaSuccess) return e;
  DecodeTcParams P;
  if (!make_pool_map_heads(&P.tmap_k, a.k_cache, a.num_blocks, a.bs_log2, a.hkv, D) ||
      !make_pool_map_heads(&P.tmap_v, a.v_cache, a.num_blocks, a.bs_log2, a.hkv, D))
    return cudaErrorInvalidValue;
  DecodeParams& p = P.p;
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
  p.fault_no_copies = a.fault == PKV_FAULT_DECODE_NO_COPIES;
  p.stream_early = a.stream_early;
  record_kernel_event(PKV_KERNEL_DECODE, false, stream);
  const cudaError_t e = launch_pdl(decode_tc_kernel<D, G, BS>, dim3(a.decode_ctas), dim3((kDecodeWarps + 1) * 32),
                                   C::kSmemBytes, stream, P);
  record_kernel_event(PKV_KERNEL_DECODE, true, stream);
  return e;
}

template <int D>
cudaError_t launch_g(const AttnArgs& a, cudaStream_t stream) {
  switch (a.hq / a.hkv) {
    case 1: return launch<D, 1>(a, stream);
    case 2: return launch<D, 2>(a, stream);
    case 3: return launch<D, 3>(a, stream);
    case 4: return launch<D, 4>(a, stream);
    case 5: return launch<D, 5>(a, stream);
    case 6: return launch<D, 6>(a, stream);
    case 7: return launch<D, 7>(a, stream);
    case 8: return launch<D, 8>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t PKV_CAT(launch_decode_tc_bs, PKV_DECODE_TC_BS)(const AttnArgs& a, cudaStream_t stream) {
  if ((1 << a.bs_log2) != BS) return cudaErrorInvalidValue;
  return a.head_dim == 128 ? launch_g<128>(a, stream) : launch_g<64>(a, stream);
}

}  // namespace pkv
