// attn_fwd_tc_rope.cu -- the tensor-core attention forward with rotary
// embedding applied inside the kernel (the kernel template is in
// attn_fwd_tc.cuh): mode 1 turns the Q rows after their load, mode 2 also the
// K rows of every key tile.  Without ALiBi; windows run on the per-unit
// kernel.
#include "attn_fwd_tc.cuh"

namespace rf {

cudaError_t launch_attn_tc_rope(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                int Hkv, int Nq, int Nk, int D, float scale, int causal, int window,
                                const float* alibi, Dt dt, unsigned* status, void* ws, int sms, int rope,
                                double rope_base, int rope_pos, cudaStream_t s) {
  AttnRope rp;
  rp.mode = rope;
  rp.base = rope_base;
  rp.pos = rope_pos;
  if (rope == 1)
    return launch_rope_mode<1>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, window, alibi, dt, status, ws,
                               sms, rp, s);
  if (rope == 2)
    return launch_rope_mode<2>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, window, alibi, dt, status, ws,
                               sms, rp, s);
  return cudaErrorNotSupported;
}

}  // namespace rf
