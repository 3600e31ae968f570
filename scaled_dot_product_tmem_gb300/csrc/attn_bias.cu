// attn_bias.cu -- launch dispatch of the additive-bias instantiations of the forward,
// kv-stationary and query-stationary backward kernels (BIAS = true): full-length and
// padded batches, (d_qk, d_v) in {(64, 64), (128, 128), (192, 128)}.  A translation
// unit of its own so that these instantiations compile in parallel with the others.
#include "attn_bwd_kernels.cuh"
#include "attn_fwd_kernel.cuh"

namespace sdpa {

// The forward's two staged bias tiles take 64 KB of shared memory: at d = 128 one K stage
// makes room for them (two V stages, so the next V load need not wait for both of this
// tile's P.V products; measured a little faster than two K stages and one V stage).
int launch_attn_fwd_bias(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, cudaStream_t stream, const CUtensorMap* tb) {
  const bool vl = p.seq_q || p.seq_kv;
  if (d_qk == 128 && d_v == 128)
    return vl ? launch_fwd_t<128, 128, 1, 2, true, false, true>(tq, tk, tv, p, stream, tb)
              : launch_fwd_t<128, 128, 1, 2, false, false, true>(tq, tk, tv, p, stream, tb);
  if (d_qk == 64 && d_v == 64)
    return vl ? launch_fwd_t<64, 64, 4, 4, true, false, true>(tq, tk, tv, p, stream, tb)
              : launch_fwd_t<64, 64, 4, 4, false, false, true>(tq, tk, tv, p, stream, tb);
  if (d_qk == 192 && d_v == 128)
    return vl ? launch_fwd_t<192, 128, 2, 1, true, false, true>(tq, tk, tv, p, stream)
              : launch_fwd_t<192, 128, 2, 1, false, false, true>(tq, tk, tv, p, stream);
  return -2;
}

int launch_bwd_kv_bias(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tb, const BwdParams& p,
                       bool fuse_dq, cudaStream_t stream) {
  constexpr KernVariant B = KernVariant::kBias;
  if (fuse_dq) {
    if (d_qk == 128 && d_v == 128) return launch_kv_t<128, 128, true, B>(tq, tk, tv, tdo, tdq, tb, p, stream);
    if (d_qk == 64 && d_v == 64) return launch_kv_t<64, 64, true, B>(tq, tk, tv, tdo, tdq, tb, p, stream);
    return -2;
  }
  if (d_qk == 128 && d_v == 128) return launch_kv_t<128, 128, false, B>(tq, tk, tv, tdo, tdq, tb, p, stream);
  if (d_qk == 64 && d_v == 64) return launch_kv_t<64, 64, false, B>(tq, tk, tv, tdo, tdq, tb, p, stream);
  if (d_qk == 192 && d_v == 128) return launch_kv_t<192, 128, false, B>(tq, tk, tv, tdo, tdq, tb, p, stream);
  return -2;
}

int launch_bwd_q_bias(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream) {
  constexpr KernVariant B = KernVariant::kBias;
  if (d_qk == 128 && d_v == 128) return launch_q_t<128, 128, B>(tq, tk, tv, tdo, p, stream);
  if (d_qk == 64 && d_v == 64) return launch_q_t<64, 64, B>(tq, tk, tv, tdo, p, stream);
  if (d_qk == 192 && d_v == 128) return launch_q_t<192, 128, B>(tq, tk, tv, tdo, p, stream);
  return -2;
}

}  // namespace sdpa
