// Internal interface between the sp_attention entry point and its kernels.
#pragma once

#include "sp_internal.cuh"

namespace sp {

struct AttnArgs {
    const void *q[SP_MAX_RANKS];
    const void *k[SP_MAX_RANKS];
    const void *v[SP_MAX_RANKS];
    void *o[SP_MAX_RANKS];
    int W, B, Tq, Tk, Hl, D;
    sp_dtype dtype;
    int64_t qs[3], ks[3], os[3];  // batch, token, head strides in elements
    // 0: q/o (resp. k/v) are per-rank [B, T, Hl, D] tensors; > 0: they are the
    // W source-rank token shards of the T = Tq (Tk) real tokens, shard_rows =
    // ceil(T / W) tokens apart: shard s holds tokens [s*shard_rows, ...) in its
    // first clamp(T - s*shard_rows, 0, shard_rows) rows, all H = W*Hl heads
    // (rank r's at [r*Hl, (r+1)*Hl)), read and written in place -- the
    // exchange fused into the attention.
    int q_shard_rows, kv_shard_rows;
    int mask_kind;
    const uint8_t *mask;
    float scale;
    WorkspaceHeader *ws;  // status word
    uint8_t *extra;       // workspace bytes after the header (split-key partials)
    size_t extra_bytes;
};

int launch_attn_simt(const AttnArgs &a, cudaStream_t st);

// Tensor-core path: bf16, D in {64, 128}, 16-byte aligned strides/pointers.
bool attn_tc_supported(const AttnArgs &a);
int launch_attn_tc(const AttnArgs &a, cudaStream_t st);
// Extra workspace bytes (beyond the header) the tensor-core path wants.
size_t attn_tc_extra_bytes(int W, int B, int Tq, int Tk, int Hl, int D);

}  // namespace sp
