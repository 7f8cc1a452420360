// Causal grouped-query attention with rotary positions (tcgen05).
//
// Layout: M rows = nseq sequences of S tokens (S % 128 == 0); q [M, H*128],
// k and v [M, Hkv*128] bf16 with row strides; query head h reads kv head
// h / (H / Hkv); positions restart at 0 in each sequence.  Scores are
// q . k / sqrt(128) with the causal mask inside each sequence.
#pragma once
#include "common.cuh"

namespace sl {

constexpr int kAtD = 128;  // head width

// table [S][128] fp32: cos(p theta^(-i/64)) at i, sin at 64 + i (i < 64).
sl_status rope_table(int64_t S, double theta, float* table, cudaStream_t stream);
// In place on x [M, nheads * 128] bf16 (row stride ld): rotate the pairs
// (i, i + 64) of every head by the row's position angle (negated: inverse).
sl_status rope_apply(uint16_t* x, int64_t ld, int64_t M, int nheads, int64_t S, const float* table, int inverse,
                     cudaStream_t stream);

struct AttnShape {
  int64_t M, S;
  int H, Hkv;
};

// o [M, H*128] bf16 (row stride ldo) and lse [H, M] fp32 (head-major: the
// natural log of the softmax normaliser of each head and row).
sl_status attention_fwd(const AttnShape& sh, const uint16_t* q, int64_t ldq, const uint16_t* k, int64_t ldk,
                        const uint16_t* v, int64_t ldv, uint16_t* o, int64_t ldo, float* lse, cudaStream_t stream);

// dq [M, H*128], dk, dv [M, Hkv*128] bf16 from o, do and lse of the forward.
// rope (nullable): a table of rope_table; dq and dk then leave rotated back
// by the inverse angle (the gradients of the unrotated q and k).  ws
// (attention_ws_bytes, 16-byte aligned): Di [H, M] and the fp32 per-head
// partials of dK and dV [H, M, 128] each.
size_t attention_ws_bytes(int64_t M, int H);
sl_status attention_bwd(const AttnShape& sh, const uint16_t* q, int64_t ldq, const uint16_t* k, int64_t ldk,
                        const uint16_t* v, int64_t ldv, const uint16_t* o, int64_t ldo, const uint16_t* dout,
                        int64_t lddo, const float* lse, uint16_t* dq, int64_t lddq, uint16_t* dk, int64_t lddk,
                        uint16_t* dv, int64_t lddv, const float* rope, void* ws, cudaStream_t stream);

}  // namespace sl
