// attn_fwd_tc.cu -- the tensor-core attention forward without rotary
// embedding (the kernel template is in attn_fwd_tc.cuh), the split-tail
// workspace size, and the dispatch of every 16-bit attention call.
#include "attn_fwd_tc.cuh"

namespace rf {

size_t attn_tc_workspace_bytes(int B, int Hq, int Nq, int Nk, int D, int causal, int sms) {
  if (causal) return 0;
  return tail_bytes(plan_for(B, Hq, Nq, Nk, sms), D);
}

cudaError_t launch_attn_tc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                           int Nq, int Nk, int D, float scale, int causal, int window, const float* alibi, Dt dt,
                           unsigned* status, void* ws, int sms, int rope, double rope_base, int rope_pos,
                           cudaStream_t s) {
  if (rope != 0)
    return launch_attn_tc_rope(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, window, alibi, dt, status, ws,
                               sms, rope, rope_base, rope_pos, s);
  // Windows of up to kWindowPersistMax keys leave units so short that the
  // persistent schedule of attn_fwd_tc_window.cu wins (measured at N = 4096:
  // W = 128 -18%, 256 -17%, 1024 -7% time; 2048 equal).
  if (causal && window > 0 && window <= kWindowPersistMax && D == 64)
    return launch_attn_tc_window(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, window, alibi, dt, status, sms, s);
  return launch_rope_mode<0>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, window, alibi, dt, status, ws, sms,
                             AttnRope{}, s);
}

}  // namespace rf
