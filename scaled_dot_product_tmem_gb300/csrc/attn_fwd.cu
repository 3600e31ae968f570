// attn_fwd.cu -- launch dispatch of the fused BSHD attention forward (the kernel is
// in attn_fwd_kernel.cuh): bf16 with full-length or padded batches, bias, E4M3.
#include "attn_fwd_kernel.cuh"

namespace sdpa {

template <bool VL>
static int launch_attn_fwd_vl(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const FwdParams& p, cudaStream_t stream) {
  if (d_qk == 128 && d_v == 128) return launch_fwd_t<128, 128, 2, 2, VL>(tq, tk, tv, p, stream);
  if (d_qk == 64 && d_v == 64) return launch_fwd_t<64, 64, 4, 4, VL>(tq, tk, tv, p, stream);
  if (d_qk == 192 && d_v == 128) return launch_fwd_t<192, 128, 2, 1, VL>(tq, tk, tv, p, stream);
  if (d_qk == 128 && d_v == 64) return launch_fwd_t<128, 64, 2, 3, VL>(tq, tk, tv, p, stream);
  if (d_qk == 64 && d_v == 128) return launch_fwd_t<64, 128, 3, 3, VL>(tq, tk, tv, p, stream);
  if (d_qk == 192 && d_v == 64) return launch_fwd_t<192, 64, 2, 2, VL>(tq, tk, tv, p, stream);
  return -2;
}

int launch_attn_fwd(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                    const FwdParams& p, cudaStream_t stream, const CUtensorMap* tb) {
  if (p.bias) return launch_attn_fwd_bias(d_qk, d_v, tq, tk, tv, p, stream, tb);  // attn_bias.cu
  // padded batches get the instantiation with the per-entry lengths and row tests
  return (p.seq_q || p.seq_kv) ? launch_attn_fwd_vl<true>(d_qk, d_v, tq, tk, tv, p, stream)
                               : launch_attn_fwd_vl<false>(d_qk, d_v, tq, tk, tv, p, stream);
}

int launch_attn_fwd_fp8(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                        const FwdParams& p, cudaStream_t stream) {
  if (d == 128) return launch_fwd_t<128, 128, 3, 3, false, true>(tq, tk, tvt, p, stream);
  if (d == 64) return launch_fwd_t<64, 64, 6, 6, false, true>(tq, tk, tvt, p, stream);
  return -2;
}

}  // namespace sdpa
