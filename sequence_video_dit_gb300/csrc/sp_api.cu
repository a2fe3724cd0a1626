// Host side of the C ABI: error reporting, device properties, and the
// sp_attention entry point (argument validation and kernel selection).
#include <math.h>
#include <atomic>
#include <mutex>
#include <stdarg.h>
#include <string.h>

#include "sp_attn.cuh"

namespace sp {

static thread_local char g_err[512] = "";
static std::atomic<uint64_t> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int set_error(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int device_info(DeviceInfo *out) {
    // per-device cache, published with release / read with acquire (callers
    // may be on several host threads; a racing first fill writes equal values)
    static DeviceInfo cache[64];
    static std::atomic<bool> have[64];
    int dev = 0;
    SP_CUDA_CHECK(cudaGetDevice(&dev));
    if (dev >= 0 && dev < 64 && have[dev].load(std::memory_order_acquire)) {
        *out = cache[dev];
        return SP_OK;
    }
    DeviceInfo d;
    d.device = dev;
    SP_CUDA_CHECK(cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev));
    SP_CUDA_CHECK(cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev));
    SP_CUDA_CHECK(cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev));
    int l2 = 0, smem = 0;
    SP_CUDA_CHECK(cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev));
    SP_CUDA_CHECK(cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
    d.l2_bytes = (size_t)l2;
    d.max_smem_optin = (size_t)smem;
    if (dev >= 0 && dev < 64 && !have[dev].load(std::memory_order_acquire)) {
        static std::mutex fill;
        std::lock_guard<std::mutex> lock(fill);
        if (!have[dev].load(std::memory_order_relaxed)) {
            cache[dev] = d;
            have[dev].store(true, std::memory_order_release);
        }
    }
    *out = d;
    return SP_OK;
}

static void default_strides(int64_t out[3], const int64_t *in, int T, int Hl, int D) {
    if (in) {
        for (int i = 0; i < 3; i++) out[i] = in[i];
    } else {
        out[2] = D;
        out[1] = (int64_t)Hl * D;
        out[0] = (int64_t)T * Hl * D;
    }
}

}  // namespace sp

using namespace sp;

extern "C" {

const char *sp_last_error(void) { return g_err; }

int sp_version(void) { return 1; }

uint64_t sp_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *sp_status_string(int status) {
    switch (status) {
        case SP_OK: return "SP_OK";
        case SP_ERR_NOT_DIVISIBLE: return "SP_ERR_NOT_DIVISIBLE";
        case SP_ERR_HEADS_NOT_DIVISIBLE: return "SP_ERR_HEADS_NOT_DIVISIBLE";
        case SP_ERR_INVALID_ARG: return "SP_ERR_INVALID_ARG";
        case SP_ERR_ALIGNMENT: return "SP_ERR_ALIGNMENT";
        case SP_ERR_UNSUPPORTED: return "SP_ERR_UNSUPPORTED";
        case SP_ERR_TIMEOUT: return "SP_ERR_TIMEOUT";
        case SP_ERR_BARRIER: return "SP_ERR_BARRIER";
        case SP_ERR_CUDA: return "SP_ERR_CUDA";
        default: return "SP_ERR_UNKNOWN";
    }
}

size_t sp_attention_workspace_bytes(int W, int B, int Tq, int Tk, int Hl, int D, sp_dtype dtype) {
    size_t extra = 0;
    if (dtype == SP_BF16 && (D == 64 || D == 128) && W >= 1 && B >= 0 && Tq >= 0 && Tk >= 0 && Hl >= 1)
        extra = attn_tc_extra_bytes(W, B, Tq, Tk, Hl, D);
    return SP_WORKSPACE_HEADER_BYTES + extra;
}

int sp_attention(const void *const *q, const void *const *k, const void *const *v, void *const *o, int W, int B,
                 int Tq, int Tk, int Hl, int D, sp_dtype dtype, const int64_t *q_strides,
                 const int64_t *kv_strides, const int64_t *o_strides, sp_mask_kind mask_kind,
                 const uint8_t *mask, float scale, void *workspace, size_t workspace_bytes, sp_stream_t stream) {
    if (W < 1 || W > SP_MAX_RANKS)
        return set_error(SP_ERR_INVALID_ARG, "sp_attention: W=%d out of [1,%d]", W, SP_MAX_RANKS);
    if (B < 0 || Tq < 0 || Tk < 0 || Hl < 1 || D < 1)
        return set_error(SP_ERR_INVALID_ARG, "sp_attention: bad sizes B=%d Tq=%d Tk=%d Hl=%d D=%d", B, Tq, Tk, Hl, D);
    if (dtype != SP_F32 && dtype != SP_BF16) return set_error(SP_ERR_UNSUPPORTED, "sp_attention: dtype %d", (int)dtype);
    if (D > 256) return set_error(SP_ERR_UNSUPPORTED, "sp_attention: D=%d > 256", D);
    if (mask_kind != SP_MASK_NONE && mask_kind != SP_MASK_KEY && mask_kind != SP_MASK_FULL)
        return set_error(SP_ERR_INVALID_ARG, "sp_attention: mask_kind %d", (int)mask_kind);
    if (mask_kind != SP_MASK_NONE && !mask && Tk > 0)
        return set_error(SP_ERR_INVALID_ARG, "sp_attention: mask is NULL");
    if (!q || !k || !v || !o) return set_error(SP_ERR_INVALID_ARG, "sp_attention: null pointer array");
    if (!workspace || workspace_bytes < SP_WORKSPACE_HEADER_BYTES)
        return set_error(SP_ERR_INVALID_ARG, "sp_attention: workspace must hold >= %d bytes", SP_WORKSPACE_HEADER_BYTES);
    if ((uintptr_t)workspace & 15) return set_error(SP_ERR_ALIGNMENT, "sp_attention: workspace not 16-byte aligned");
    AttnArgs a;
    memset(&a, 0, sizeof(a));
    a.W = W;
    a.B = B;
    a.Tq = Tq;
    a.Tk = Tk;
    a.Hl = Hl;
    a.D = D;
    a.dtype = dtype;
    default_strides(a.qs, q_strides, Tq, Hl, D);
    default_strides(a.ks, kv_strides, Tk, Hl, D);
    default_strides(a.os, o_strides, Tq, Hl, D);
    const size_t elt = dtype == SP_F32 ? 4 : 2;
    if ((int64_t)W * B * Hl * Tq == 0) return SP_OK;  // nothing to compute (empty tensors may be null)
    for (int r = 0; r < W; r++) {
        if (!q[r] || !o[r] || (Tk > 0 && (!k[r] || !v[r])))
            return set_error(SP_ERR_INVALID_ARG, "sp_attention: null tensor for rank %d", r);
        if (((uintptr_t)q[r] | (uintptr_t)k[r] | (uintptr_t)v[r] | (uintptr_t)o[r]) % elt)
            return set_error(SP_ERR_ALIGNMENT, "sp_attention: tensor of rank %d not element-aligned", r);
        a.q[r] = q[r];
        a.k[r] = k[r];
        a.v[r] = v[r];
        a.o[r] = o[r];
    }
    a.mask_kind = mask_kind;
    a.mask = mask;
    a.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
    a.ws = (WorkspaceHeader *)workspace;
    a.extra = (uint8_t *)workspace + SP_WORKSPACE_HEADER_BYTES;
    a.extra_bytes = workspace_bytes - SP_WORKSPACE_HEADER_BYTES;
    cudaStream_t st = (cudaStream_t)stream;
    if ((int64_t)W * B * Hl * Tq == 0) return SP_OK;
    if (attn_tc_supported(a)) return launch_attn_tc(a, st);
    return launch_attn_simt(a, st);
}

int sp_attention_shards(const void *const *q, const void *const *k, const void *const *v, void *const *o, int W,
                        int B, int Tq, int Tk, int H, int D, sp_dtype dtype, int shard_flags,
                        const int64_t *q_strides, const int64_t *kv_strides, const int64_t *o_strides,
                        sp_mask_kind mask_kind, const uint8_t *mask, float scale, void *workspace,
                        size_t workspace_bytes, sp_stream_t stream) {
    if (W < 1 || W > SP_MAX_RANKS)
        return set_error(SP_ERR_INVALID_ARG, "sp_attention_shards: W=%d out of [1,%d]", W, SP_MAX_RANKS);
    if (B < 0 || Tq < 0 || Tk < 0 || H < 1 || D < 1)
        return set_error(SP_ERR_INVALID_ARG, "sp_attention_shards: bad sizes B=%d Tq=%d Tk=%d H=%d D=%d", B, Tq, Tk,
                         H, D);
    if (shard_flags & ~(SP_SHARD_Q | SP_SHARD_KV))
        return set_error(SP_ERR_INVALID_ARG, "sp_attention_shards: shard_flags %d", shard_flags);
    if (H % W != 0)
        return set_error(SP_ERR_HEADS_NOT_DIVISIBLE, "sp_attention_shards: H=%d is not divisible by W=%d", H, W);
    const bool sq = (shard_flags & SP_SHARD_Q) != 0, skv = (shard_flags & SP_SHARD_KV) != 0;
    // a sharded operand of T tokens: shards of Tl = ceil(T / W) tokens, the
    // last ones short of real rows when T % W != 0 (the pages' padded
    // partition; pad rows need not exist)
    const int q_tl = sq ? (int)(((int64_t)Tq + W - 1) / W) : 0, kv_tl = skv ? (int)(((int64_t)Tk + W - 1) / W) : 0;
    if (dtype != SP_BF16 || (D != 64 && D != 128))
        return set_error(SP_ERR_UNSUPPORTED, "sp_attention_shards: bf16 with D = 64 or 128 only");
    if (mask_kind != SP_MASK_NONE && mask_kind != SP_MASK_KEY && mask_kind != SP_MASK_FULL)
        return set_error(SP_ERR_INVALID_ARG, "sp_attention_shards: mask_kind %d", (int)mask_kind);
    if (mask_kind != SP_MASK_NONE && !mask && Tk > 0)
        return set_error(SP_ERR_INVALID_ARG, "sp_attention_shards: mask is NULL");
    if (!q || !k || !v || !o) return set_error(SP_ERR_INVALID_ARG, "sp_attention_shards: null pointer array");
    if (!workspace || workspace_bytes < SP_WORKSPACE_HEADER_BYTES)
        return set_error(SP_ERR_INVALID_ARG, "sp_attention_shards: workspace must hold >= %d bytes",
                         SP_WORKSPACE_HEADER_BYTES);
    if ((uintptr_t)workspace & 15)
        return set_error(SP_ERR_ALIGNMENT, "sp_attention_shards: workspace not 16-byte aligned");
    AttnArgs a;
    memset(&a, 0, sizeof(a));
    a.W = W;
    a.B = B;
    a.Tq = Tq;
    a.Tk = Tk;
    a.Hl = H / W;
    a.D = D;
    a.dtype = dtype;
    a.q_shard_rows = q_tl;
    a.kv_shard_rows = kv_tl;
    default_strides(a.qs, q_strides, sq ? q_tl : Tq, sq ? H : a.Hl, D);
    default_strides(a.ks, kv_strides, skv ? kv_tl : Tk, skv ? H : a.Hl, D);
    default_strides(a.os, o_strides, sq ? q_tl : Tq, sq ? H : a.Hl, D);
    if ((int64_t)W * B * (H / W) * Tq == 0) return SP_OK;  // nothing to compute (empty tensors may be null)
    for (int r = 0; r < W; r++) {
        // a shard with no real rows is never read and may be NULL
        const bool need_q = !sq || (int64_t)r * q_tl < Tq, need_kv = Tk > 0 && (!skv || (int64_t)r * kv_tl < Tk);
        if ((need_q && (!q[r] || !o[r])) || (need_kv && (!k[r] || !v[r])))
            return set_error(SP_ERR_INVALID_ARG, "sp_attention_shards: null tensor %d", r);
        a.q[r] = q[r];
        a.k[r] = k[r];
        a.v[r] = v[r];
        a.o[r] = o[r];
    }
    a.mask_kind = mask_kind;
    a.mask = mask;
    a.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
    a.ws = (WorkspaceHeader *)workspace;
    a.extra = (uint8_t *)workspace + SP_WORKSPACE_HEADER_BYTES;
    a.extra_bytes = workspace_bytes - SP_WORKSPACE_HEADER_BYTES;
    if ((int64_t)W * B * a.Hl * Tq == 0) return SP_OK;
    if (Tk == 0) return set_error(SP_ERR_UNSUPPORTED, "sp_attention_shards: no keys");
    if (!attn_tc_supported(a))
        return set_error(SP_ERR_ALIGNMENT, "sp_attention_shards: tensors and strides must be 16-byte aligned");
    return launch_attn_tc(a, (cudaStream_t)stream);
}

}  // extern "C"
