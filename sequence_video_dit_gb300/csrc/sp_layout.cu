// Layout kernels of the sequence-parallel step: pad, padding masks, tile,
// the token x head exchange (send_recv_heads / gather_heads) with SM rotation
// and per-destination completion counters, gather_output and unpad.
//
// Source: "LTX-2 序列并行拆解" (LTX-2 sequence-parallel breakdown), sections
// 补齐 (pad), 切分 (partition), 换头 (head exchange), 还原 (restore), and the
// kernel paragraphs "SM 轮转" (SM rotation) and "barrier".
//
// All of these are pure data movement and bound by HBM bandwidth.  Each kernel
// walks "rows" (a token's contiguous run of bytes); a group of `tx` lanes
// (a power of two <= 32) copies one row with the widest vector the pointers
// and sizes allow (16 bytes on every workload of interest), four vectors in
// flight per lane.  Index arithmetic happens once per row, not per vector.
#include <stdarg.h>
#include <string.h>

#include <mutex>

#include "sp_internal.cuh"

namespace sp {

template <int V> struct VecT;
template <> struct VecT<16> { using T = uint4; };
template <> struct VecT<8> { using T = uint2; };
template <> struct VecT<4> { using T = uint32_t; };
template <> struct VecT<2> { using T = uint16_t; };
template <> struct VecT<1> { using T = uint8_t; };

template <int V>
__device__ __forceinline__ typename VecT<V>::T vzero() {
    typename VecT<V>::T z;
    memset(&z, 0, sizeof(z));
    return z;
}

// Copy (src != nullptr) or zero-fill (src == nullptr) `nvec` vectors; the
// lanes of a group stride by `tx`.
template <int V>
__device__ __forceinline__ void copy_row(uint8_t *__restrict__ dst, const uint8_t *__restrict__ src,
                                         int nvec, int lane, int tx) {
    using T = typename VecT<V>::T;
    T *d = reinterpret_cast<T *>(dst);
    if (src == nullptr) {
        const T z = vzero<V>();
        for (int i = lane; i < nvec; i += tx) d[i] = z;
        return;
    }
    const T *s = reinterpret_cast<const T *>(src);
    int i = lane;
    for (; i + 3 * tx < nvec; i += 4 * tx) {
        T a0 = s[i], a1 = s[i + tx], a2 = s[i + 2 * tx], a3 = s[i + 3 * tx];
        d[i] = a0;
        d[i + tx] = a1;
        d[i + 2 * tx] = a2;
        d[i + 3 * tx] = a3;
    }
    // At most three vectors per lane are left.  Their loads are all issued
    // before the first store: a 1 KB exchange piece is exactly this tail (two
    // vectors per lane), and a load-store-load-store order there halves the
    // loads in flight (measured: 0.77 -> 0.92 of the copy bandwidth at 403 MB).
    const bool h0 = i < nvec, h1 = i + tx < nvec, h2 = i + 2 * tx < nvec;
    T a0 = vzero<V>(), a1 = vzero<V>(), a2 = vzero<V>();
    if (h0) a0 = s[i];
    if (h1) a1 = s[i + tx];
    if (h2) a2 = s[i + 2 * tx];
    if (h0) d[i] = a0;
    if (h1) d[i + tx] = a1;
    if (h2) d[i + 2 * tx] = a2;
}

// ---------------------------------------------------------------- row ops
struct PadOp {  // x [B,T,rb] -> y [B,T_pad,rb], zero rows for t >= T
    const uint8_t *x;
    uint8_t *y;
    int T, T_pad;
    int64_t rb;
    __device__ void row(uint32_t r, const uint8_t *&src, uint8_t *&dst) const {
        uint32_t b = r / (uint32_t)T_pad, t = r - b * (uint32_t)T_pad;
        dst = y + (int64_t)r * rb;
        src = (t < (uint32_t)T) ? x + ((int64_t)b * T + t) * rb : nullptr;
    }
};

struct UnpadOp {  // x [B,T_pad,rb] -> y [B,T,rb]
    const uint8_t *x;
    uint8_t *y;
    int T, T_pad;
    int64_t rb;
    __device__ void row(uint32_t r, const uint8_t *&src, uint8_t *&dst) const {
        uint32_t b = r / (uint32_t)T, t = r - b * (uint32_t)T;
        dst = y + (int64_t)r * rb;
        src = x + ((int64_t)b * T_pad + t) * rb;
    }
};

struct TileOp {  // x [B,T_pad,rb] -> shard[r] [B,Tl,rb]; rows enumerate (r, b, t)
    const uint8_t *x;
    uint8_t *shard[SP_MAX_RANKS];
    int B, Tl, T_pad;
    int64_t rb;
    __device__ void row(uint32_t i, const uint8_t *&src, uint8_t *&dst) const {
        uint32_t per_rank = (uint32_t)B * Tl;
        uint32_t r = i / per_rank, j = i - r * per_rank;
        uint32_t b = j / (uint32_t)Tl, t = j - b * (uint32_t)Tl;
        dst = shard[r] + (int64_t)j * rb;
        src = x + ((int64_t)b * T_pad + (int64_t)r * Tl + t) * rb;
    }
};

struct GatherOutOp {  // shard[r] [B,Tl,rb] -> y [B,T_out,rb]; token g comes from rank g / Tl
    const uint8_t *shard[SP_MAX_RANKS];
    uint8_t *y;
    int Tl, T_out;
    int64_t rb;
    __device__ void row(uint32_t i, const uint8_t *&src, uint8_t *&dst) const {
        uint32_t b = i / (uint32_t)T_out, g = i - b * (uint32_t)T_out;
        uint32_t r = g / (uint32_t)Tl, t = g - r * (uint32_t)Tl;
        dst = y + (int64_t)i * rb;
        src = shard[r] + ((int64_t)b * Tl + t) * rb;
    }
};

// 2-D spatial split of the latent grid (LongCat-Video context parallel):
// x [B, F, Hg, Wg, rb] <-> shard[ih*sw + iw] [B, F, bh, bw, rb] with
// bh = Hg / sh, bw = Wg / sw.  Rows enumerate (rank, b, f, h, w) so the shard
// side is contiguous and the grid side is read or written in runs of bw rows.
template <bool GATHER>
struct Split2DOp {
    uint8_t *grid;  // source (tile) or destination (gather)
    uint8_t *shard[SP_MAX_RANKS];
    uint32_t per_rank;  // B * F * bh * bw
    uint32_t bh, bw, Hg, Wg, sw;
    int64_t rb;
    __device__ void row(uint32_t i, const uint8_t *&src, uint8_t *&dst) const {
        const uint32_t r = i / per_rank, j = i - r * per_rank;
        const uint32_t jw = j / bw, w = j - jw * bw;
        const uint32_t bf = jw / bh, h = jw - bf * bh;  // bf = b * F + f
        const uint32_t ih = r / sw, iw = r - ih * sw;
        const int64_t g = ((int64_t)bf * Hg + (int64_t)ih * bh + h) * Wg + (int64_t)iw * bw + w;
        uint8_t *sp = shard[r] + (int64_t)j * rb;
        uint8_t *gp = grid + g * rb;
        if (GATHER) {
            src = sp;
            dst = gp;
        } else {
            src = gp;
            dst = sp;
        }
    }
};

template <int V, class Op>
__global__ void __launch_bounds__(256) rows_kernel(Op op, uint32_t nrows, int nvec, int tx_log2) {
    const int tx = 1 << tx_log2;
    const int lane = threadIdx.x & (tx - 1);
    const uint32_t group = (blockIdx.x * blockDim.x + threadIdx.x) >> tx_log2;
    const uint32_t ngroups = (gridDim.x * blockDim.x) >> tx_log2;
    for (uint32_t r = group; r < nrows; r += ngroups) {
        const uint8_t *src;
        uint8_t *dst;
        op.row(r, src, dst);
        copy_row<V>(dst, src, nvec, lane, tx);
    }
}

static int tx_log2_for(int nvec) {
    int l = 0;
    while (l < 5 && (1 << l) < nvec) l++;
    return l;
}

template <class Op>
static int launch_rows(const Op &op, uint64_t nrows, int64_t row_bytes, int V, cudaStream_t st,
                       const char *what) {
    if (nrows == 0 || row_bytes == 0) return SP_OK;
    if (nrows > 0x7fffffffull) return set_error(SP_ERR_INVALID_ARG, "%s: too many rows", what);
    if (row_bytes / V > 0x7fffffff) return set_error(SP_ERR_INVALID_ARG, "%s: row too long", what);
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    const int nvec = (int)(row_bytes / V);
    const int tl = tx_log2_for(nvec);
    const int threads = 256;
    uint64_t want = (nrows * (uint64_t)(1 << tl) + threads - 1) / threads;
    uint64_t cap = (uint64_t)di.num_sms * 8;
    unsigned grid = (unsigned)(want < cap ? want : cap);
    if (grid == 0) grid = 1;
    switch (V) {
        case 16: rows_kernel<16, Op><<<grid, threads, 0, st>>>(op, (uint32_t)nrows, nvec, tl); break;
        case 8: rows_kernel<8, Op><<<grid, threads, 0, st>>>(op, (uint32_t)nrows, nvec, tl); break;
        case 4: rows_kernel<4, Op><<<grid, threads, 0, st>>>(op, (uint32_t)nrows, nvec, tl); break;
        case 2: rows_kernel<2, Op><<<grid, threads, 0, st>>>(op, (uint32_t)nrows, nvec, tl); break;
        default: rows_kernel<1, Op><<<grid, threads, 0, st>>>(op, (uint32_t)nrows, nvec, tl); break;
    }
    return check_launch(what);
}

// ---------------------------------------------------------------- masks
__global__ void pad_mask_key_kernel(uint8_t *out, int T, int T_pad) {
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < T_pad; k += gridDim.x * blockDim.x)
        out[k] = (k < T) ? 1 : 0;
}

// One warp per (b, q) row of the extended (B, T_pad, T_pad) mask.
__global__ void pad_mask_user_kernel(const uint8_t *__restrict__ user, uint8_t *__restrict__ out,
                                     int B, int T, int T_pad) {
    const int lane = threadIdx.x & 31;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    const uint32_t nrows = (uint32_t)B * T_pad;
    for (uint32_t row = warp; row < nrows; row += nwarps) {
        const uint32_t b = row / (uint32_t)T_pad, q = row - b * (uint32_t)T_pad;
        uint8_t *o = out + (int64_t)row * T_pad;
        const uint8_t *u = user + ((int64_t)b * T + q) * T;
        for (int k = lane; k < T_pad; k += 32) {
            uint8_t m;
            if (k >= T) m = 0;
            else if (q >= (uint32_t)T) m = 1;
            else m = u[k] ? 1 : 0;
            o[k] = m;
        }
    }
}

// ---------------------------------------------------------------- exchange
struct ExchangeParams {
    const uint8_t *src[SP_MAX_RANKS];
    uint8_t *dst[SP_MAX_RANKS];
    int W, Tl;
    uint32_t chunks_per_rank;  // B * W * Tl
    uint32_t T_all;            // W * Tl
    int64_t chunk_bytes;       // Hl * D * elt
    int64_t row_bytes;         // H * D * elt
    WorkspaceHeader *ws;
};

// Completion barrier ("barrier" paragraph): make this CTA's writes visible,
// then count it on its destination rank.  The last CTA to take a ticket checks
// every counter against the CTA map, records the counts and resets them.
__device__ __forceinline__ void exchange_complete(WorkspaceHeader *ws, int r, int W) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0 && ws != nullptr) {
        atomicAdd(&ws->counters[r], 1);
        __threadfence();
        const int ticket = atomicAdd(&ws->ticket, 1);
        if (ticket == (int)gridDim.x - 1) {
            __threadfence();
            for (int q = 0; q < SP_MAX_RANKS; q++) {
                const int seen = atomicExch(&ws->counters[q], 0);
                const int expect = q < W ? (int)((gridDim.x - q + W - 1) / W) : 0;
                ws->observed[q] = seen;
                if (seen != expect) set_device_status(&ws->status, SP_ERR_BARRIER);
            }
            ws->grid = (int)gridDim.x;
            atomicAdd(&ws->launches, 1);
            __threadfence();
            atomicExch(&ws->ticket, 0);
        }
    }
}

// GATHER = false: send_recv_heads.  CTA i serves rank r = i % W (SM rotation)
// and its rank group walks r's chunks c = (b, s*Tl + t) with a stride; the
// destination heads[r] + c*chunk is contiguous, the source is the r-th head
// block of token t of shard s.  GATHER = true moves the same chunks back.
template <int V, bool GATHER>
__global__ void __launch_bounds__(256) exchange_kernel(ExchangeParams p, int nvec, int tx_log2) {
    const int W = p.W;
    const int r = blockIdx.x % W;
    const uint32_t g = blockIdx.x / W;
    const uint32_t n_r = (gridDim.x - r + W - 1) / W;  // CTAs serving rank r
    const int tx = 1 << tx_log2;
    const int lane = threadIdx.x & (tx - 1);
    const uint32_t groups_per_cta = blockDim.x >> tx_log2;
    const uint32_t gid = g * groups_per_cta + (threadIdx.x >> tx_log2);
    const uint32_t ngroups = n_r * groups_per_cta;
    uint8_t *const heads_r = GATHER ? nullptr : p.dst[r];
    const uint8_t *const heads_src_r = GATHER ? p.src[r] : nullptr;
    for (uint32_t c = gid; c < p.chunks_per_rank; c += ngroups) {
        const uint32_t b = c / p.T_all, tg = c - b * p.T_all;
        const uint32_t s = tg / (uint32_t)p.Tl, t = tg - s * (uint32_t)p.Tl;
        const int64_t tok_off = ((int64_t)b * p.Tl + t) * p.row_bytes + (int64_t)r * p.chunk_bytes;
        if (!GATHER) {
            copy_row<V>(heads_r + (int64_t)c * p.chunk_bytes, p.src[s] + tok_off, nvec, lane, tx);
        } else {
            copy_row<V>(p.dst[s] + tok_off, heads_src_r + (int64_t)c * p.chunk_bytes, nvec, lane, tx);
        }
    }
    exchange_complete(p.ws, r, W);
}

// The exchange fused with its neighbours, for a caller-held [B, T, H, D]
// tensor x (one GPU: the token shards never need to exist).
//   GATHER = false  (pad + tile + send_recv_heads):
//     heads[r][b, g, h', :] = g < T ? x[b, g, r*Hl + h', :] : 0,   g < T_pad
//   GATHER = true   (gather_heads + gather_output cropped to T_out):
//     y[b, g, r*Hl + h', :] = heads[r][b, g, h', :],               g < T_out
// Same SM rotation, chunk walk and completion barrier as exchange_kernel.
struct FusedParams {
    uint8_t *heads[SP_MAX_RANKS];
    uint8_t *x;         // caller tensor: source (send) or destination (gather)
    int W, T_real;      // T_real = T (send) or T_out (gather)
    uint32_t T_pad;
    uint32_t chunks_per_rank;  // B * T_pad
    int64_t chunk_bytes, row_bytes;
    WorkspaceHeader *ws;
};

template <int V, bool GATHER>
__global__ void __launch_bounds__(256) exchange_fused_kernel(FusedParams p, int nvec, int tx_log2) {
    const int W = p.W;
    const int r = blockIdx.x % W;
    const uint32_t grp = blockIdx.x / W;
    const uint32_t n_r = (gridDim.x - r + W - 1) / W;
    const int tx = 1 << tx_log2;
    const int lane = threadIdx.x & (tx - 1);
    const uint32_t groups_per_cta = blockDim.x >> tx_log2;
    const uint32_t gid = grp * groups_per_cta + (threadIdx.x >> tx_log2);
    const uint32_t ngroups = n_r * groups_per_cta;
    uint8_t *const heads_r = p.heads[r];
    for (uint32_t c = gid; c < p.chunks_per_rank; c += ngroups) {
        const uint32_t b = c / p.T_pad, g = c - b * p.T_pad;
        const bool real = g < (uint32_t)p.T_real;
        const int64_t x_off = ((int64_t)b * p.T_real + g) * p.row_bytes + (int64_t)r * p.chunk_bytes;
        if (!GATHER) {
            copy_row<V>(heads_r + (int64_t)c * p.chunk_bytes, real ? p.x + x_off : nullptr, nvec, lane, tx);
        } else if (real) {
            copy_row<V>(p.x + x_off, heads_r + (int64_t)c * p.chunk_bytes, nvec, lane, tx);
        }
    }
    exchange_complete(p.ws, r, W);
}

static int exchange_grid(const DeviceInfo &di) { return di.num_sms * 4; }

template <bool GATHER>
static int launch_exchange_fused(void *x, void *const *heads, int W, int B, int T_pad, int T_real, int H, int D,
                                 int elt, void *workspace, cudaStream_t st, const char *what) {
    if (W < 1 || W > SP_MAX_RANKS) return set_error(SP_ERR_INVALID_ARG, "%s: W=%d out of [1,%d]", what, W, SP_MAX_RANKS);
    if (B < 0 || T_pad < 0 || T_real < 0 || T_real > T_pad || H < 1 || D < 1)
        return set_error(SP_ERR_INVALID_ARG, "%s: bad sizes", what);
    if (elt != 1 && elt != 2 && elt != 4 && elt != 8) return set_error(SP_ERR_INVALID_ARG, "%s: elt_bytes=%d", what, elt);
    if (T_pad % W != 0)
        return set_error(SP_ERR_NOT_DIVISIBLE, "total_tokens=%d is not divisible by world_size=%d", T_pad, W);
    if (H % W != 0) return set_error(SP_ERR_HEADS_NOT_DIVISIBLE, "%s: H=%d is not divisible by W=%d", what, H, W);
    if (!heads || !workspace) return set_error(SP_ERR_INVALID_ARG, "%s: null pointer array or workspace", what);
    if (((uintptr_t)workspace & 15) != 0) return set_error(SP_ERR_ALIGNMENT, "%s: workspace not 16-byte aligned", what);
    const int Hl = H / W;
    FusedParams p;
    memset(&p, 0, sizeof(p));
    p.chunk_bytes = (int64_t)Hl * D * elt;
    p.row_bytes = (int64_t)H * D * elt;
    uint64_t align = (uint64_t)p.chunk_bytes;
    const bool any = (int64_t)B * T_pad > 0;
    if (any && T_real > 0 && !x) return set_error(SP_ERR_INVALID_ARG, "%s: null tensor", what);
    p.x = (uint8_t *)x;
    align |= (uint64_t)(uintptr_t)x;
    for (int i = 0; i < W; i++) {
        if (any && !heads[i]) return set_error(SP_ERR_INVALID_ARG, "%s: null buffer for rank %d", what, i);
        p.heads[i] = (uint8_t *)heads[i];
        align |= (uint64_t)(uintptr_t)heads[i];
    }
    const int V = vector_width(align ? align : 16);
    p.W = W;
    p.T_real = T_real;
    p.T_pad = (uint32_t)T_pad;
    const uint64_t chunks = (uint64_t)B * T_pad;
    if (chunks > 0x7fffffffull) return set_error(SP_ERR_INVALID_ARG, "%s: too many tokens", what);
    p.chunks_per_rank = (uint32_t)chunks;
    p.ws = (WorkspaceHeader *)workspace;
    if (chunks == 0) return SP_OK;
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    const int nvec = (int)(p.chunk_bytes / V);
    const int tl = tx_log2_for(nvec);
    int grid = exchange_grid(di);
    if (grid < W) grid = W;
    switch (V) {
        case 16: exchange_fused_kernel<16, GATHER><<<grid, 256, 0, st>>>(p, nvec, tl); break;
        case 8: exchange_fused_kernel<8, GATHER><<<grid, 256, 0, st>>>(p, nvec, tl); break;
        case 4: exchange_fused_kernel<4, GATHER><<<grid, 256, 0, st>>>(p, nvec, tl); break;
        case 2: exchange_fused_kernel<2, GATHER><<<grid, 256, 0, st>>>(p, nvec, tl); break;
        default: exchange_fused_kernel<1, GATHER><<<grid, 256, 0, st>>>(p, nvec, tl); break;
    }
    return check_launch(what);
}

// Host-side checks and kernel parameters of one exchange (nothing is issued).
static int prepare_exchange(const void *const *src, void *const *dst, int W, int B, int Tl, int H, int D, int elt,
                            void *workspace, const char *what, ExchangeParams &p, int &V) {
    if (W < 1 || W > SP_MAX_RANKS) return set_error(SP_ERR_INVALID_ARG, "%s: W=%d out of [1,%d]", what, W, SP_MAX_RANKS);
    if (B < 0 || Tl < 0 || H < 1 || D < 1) return set_error(SP_ERR_INVALID_ARG, "%s: bad sizes", what);
    if (elt != 1 && elt != 2 && elt != 4 && elt != 8) return set_error(SP_ERR_INVALID_ARG, "%s: elt_bytes=%d", what, elt);
    if (H % W != 0) return set_error(SP_ERR_HEADS_NOT_DIVISIBLE, "%s: H=%d is not divisible by W=%d", what, H, W);
    if (!src || !dst || !workspace) return set_error(SP_ERR_INVALID_ARG, "%s: null pointer array or workspace", what);
    if (((uintptr_t)workspace & 15) != 0) return set_error(SP_ERR_ALIGNMENT, "%s: workspace not 16-byte aligned", what);
    const int Hl = H / W;
    memset(&p, 0, sizeof(p));
    uint64_t align = 0;
    p.chunk_bytes = (int64_t)Hl * D * elt;
    p.row_bytes = (int64_t)H * D * elt;
    align |= (uint64_t)p.chunk_bytes;
    const bool any = (int64_t)B * Tl > 0;  // empty tensors may carry null pointers
    for (int i = 0; i < W; i++) {
        if (any && (!src[i] || !dst[i])) return set_error(SP_ERR_INVALID_ARG, "%s: null buffer for rank %d", what, i);
        p.src[i] = (const uint8_t *)src[i];
        p.dst[i] = (uint8_t *)dst[i];
        align |= (uint64_t)(uintptr_t)src[i] | (uint64_t)(uintptr_t)dst[i];
    }
    V = vector_width(align ? align : 16);
    p.W = W;
    p.Tl = Tl;
    p.T_all = (uint32_t)W * Tl;
    uint64_t chunks = (uint64_t)B * W * Tl;
    if (chunks > 0x7fffffffull) return set_error(SP_ERR_INVALID_ARG, "%s: too many tokens", what);
    p.chunks_per_rank = (uint32_t)chunks;
    p.ws = (WorkspaceHeader *)workspace;
    return SP_OK;
}

template <bool GATHER>
static int run_exchange(const ExchangeParams &p, int V, cudaStream_t st, const char *what) {
    if (p.chunks_per_rank == 0) return SP_OK;
    const int W = p.W;
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    const int nvec = (int)(p.chunk_bytes / V);
    const int tl = tx_log2_for(nvec);
    int grid = exchange_grid(di);
    if (grid < W) grid = W;
    switch (V) {
        case 16: exchange_kernel<16, GATHER><<<grid, 256, 0, st>>>(p, nvec, tl); break;
        case 8: exchange_kernel<8, GATHER><<<grid, 256, 0, st>>>(p, nvec, tl); break;
        case 4: exchange_kernel<4, GATHER><<<grid, 256, 0, st>>>(p, nvec, tl); break;
        case 2: exchange_kernel<2, GATHER><<<grid, 256, 0, st>>>(p, nvec, tl); break;
        default: exchange_kernel<1, GATHER><<<grid, 256, 0, st>>>(p, nvec, tl); break;
    }
    return check_launch(what);
}

template <bool GATHER>
static int launch_exchange(const void *const *src, void *const *dst, int W, int B, int Tl, int H,
                           int D, int elt, void *workspace, cudaStream_t st, const char *what) {
    ExchangeParams p;
    int V = 16;
    int rc = prepare_exchange(src, dst, W, B, Tl, H, D, elt, workspace, what, p, V);
    if (rc) return rc;
    return run_exchange<GATHER>(p, V, st, what);
}

// ---------------------------------------------------------------- allocation-free exchange
// Scratch of sp_send_recv_heads_noalloc: one exchange header (status word,
// finish ticket, SP_MAX_RANKS completion counters) in static device memory,
// so callers that cannot allocate device memory still get the exchange.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SP_WORKSPACE_HEADER_BYTES];

// Device address of g_noalloc_scratch per device, looked up on the first call
// made with that device current.  In host code the symbol names a host-side
// stand-in, never the device memory, so only this address is passed on.
static std::mutex g_noalloc_mu;
static void *g_noalloc_addr[64];

static int noalloc_scratch(void **out) {
    int dev = 0;
    SP_CUDA_CHECK(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return set_error(SP_ERR_INVALID_ARG, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return set_error(SP_ERR_CUDA, "cudaGetSymbolAddress of the exchange scratch failed: %s",
                             cudaGetErrorString(e));
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return SP_OK;
}

template <bool GATHER>
static int launch_split_2d(const void *grid, const void *const *shards, int B, int F, int Hg, int Wg, int sh, int sw,
                           int64_t row_bytes, cudaStream_t st, const char *what) {
    if (B < 0 || F < 0 || Hg < 0 || Wg < 0 || row_bytes < 0 || !shards || sh < 1 || sw < 1 ||
        (int64_t)sh * sw > SP_MAX_RANKS)
        return set_error(SP_ERR_INVALID_ARG, "%s: bad args (split %dx%d, at most %d ranks)", what, sh, sw,
                         SP_MAX_RANKS);
    if (Hg % sh != 0 || Wg % sw != 0)
        return set_error(SP_ERR_NOT_DIVISIBLE, "%s: grid %dx%d is not divisible by the split %dx%d", what, Hg, Wg,
                         sh, sw);
    const int W = sh * sw;
    const uint64_t rows = (uint64_t)B * F * Hg * Wg;
    if (rows > 0x7fffffffull) return set_error(SP_ERR_INVALID_ARG, "%s: too many tokens", what);
    Split2DOp<GATHER> op;
    memset(&op, 0, sizeof(op));
    op.grid = (uint8_t *)grid;
    op.bh = (uint32_t)(Hg / sh);
    op.bw = (uint32_t)(Wg / sw);
    op.Hg = (uint32_t)Hg;
    op.Wg = (uint32_t)Wg;
    op.sw = (uint32_t)sw;
    op.per_rank = (uint32_t)(rows / W);
    op.rb = row_bytes;
    const bool any = rows > 0 && row_bytes > 0;
    if (any && !grid) return set_error(SP_ERR_INVALID_ARG, "%s: null grid tensor", what);
    uint64_t align = (uint64_t)(uintptr_t)grid | (uint64_t)row_bytes;
    for (int r = 0; r < W; r++) {
        if (any && !shards[r]) return set_error(SP_ERR_INVALID_ARG, "%s: null shard %d", what, r);
        op.shard[r] = (uint8_t *)shards[r];
        align |= (uint64_t)(uintptr_t)shards[r];
    }
    return launch_rows(op, rows, row_bytes, vector_width(align), st, what);
}

}  // namespace sp

using namespace sp;

extern "C" {

int sp_padded_len(int T, int W, int *T_pad) {
    if (T < 0 || W < 1 || !T_pad) return set_error(SP_ERR_INVALID_ARG, "sp_padded_len: T=%d W=%d", T, W);
    *T_pad = (int)(((int64_t)T + W - 1) / W * W);
    return SP_OK;
}

int sp_partition(int total_tokens, int W, int *starts, int *lens) {
    if (total_tokens < 0 || W < 1 || !starts || !lens)
        return set_error(SP_ERR_INVALID_ARG, "sp_partition: total=%d W=%d", total_tokens, W);
    if (total_tokens % W != 0)
        return set_error(SP_ERR_NOT_DIVISIBLE, "total_tokens=%d is not divisible by world_size=%d",
                         total_tokens, W);
    const int Tl = total_tokens / W;
    for (int r = 0; r < W; r++) {
        starts[r] = r * Tl;
        lens[r] = Tl;
    }
    return SP_OK;
}

int sp_sm_rotation_counts(int n_ctas, int W, int *counts) {
    if (n_ctas < 0 || W < 1 || !counts) return set_error(SP_ERR_INVALID_ARG, "sp_sm_rotation_counts: bad args");
    for (int r = 0; r < W; r++) counts[r] = (n_ctas - r + W - 1) / W;
    return SP_OK;
}

int sp_exchange_grid(int *n_ctas) {
    if (!n_ctas) return set_error(SP_ERR_INVALID_ARG, "sp_exchange_grid: null");
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    *n_ctas = exchange_grid(di);
    return SP_OK;
}

int sp_pad(const void *x, void *x_pad, int B, int T, int T_pad, int64_t row_bytes, sp_stream_t stream) {
    if (B < 0 || T < 0 || T_pad < T || row_bytes < 0) return set_error(SP_ERR_INVALID_ARG, "sp_pad: bad sizes");
    if ((!x && (int64_t)B * T * row_bytes > 0) || (!x_pad && (int64_t)B * T_pad * row_bytes > 0))
        return set_error(SP_ERR_INVALID_ARG, "sp_pad: null pointer");
    PadOp op{(const uint8_t *)x, (uint8_t *)x_pad, T, T_pad, row_bytes};
    int V = vector_width((uint64_t)(uintptr_t)x | (uint64_t)(uintptr_t)x_pad | (uint64_t)row_bytes);
    return launch_rows(op, (uint64_t)B * T_pad, row_bytes, V, (cudaStream_t)stream, "sp_pad");
}

int sp_unpad(const void *x_pad, void *out, int B, int T_pad, int T, int64_t row_bytes, sp_stream_t stream) {
    if (B < 0 || T < 0 || T_pad < T || row_bytes < 0) return set_error(SP_ERR_INVALID_ARG, "sp_unpad: bad sizes");
    if ((!x_pad || !out) && (int64_t)B * T * row_bytes > 0) return set_error(SP_ERR_INVALID_ARG, "sp_unpad: null pointer");
    UnpadOp op{(const uint8_t *)x_pad, (uint8_t *)out, T, T_pad, row_bytes};
    int V = vector_width((uint64_t)(uintptr_t)x_pad | (uint64_t)(uintptr_t)out | (uint64_t)row_bytes);
    return launch_rows(op, (uint64_t)B * T, row_bytes, V, (cudaStream_t)stream, "sp_unpad");
}

int sp_pad_mask(const uint8_t *user_mask, uint8_t *mask_out, int B, int T, int T_pad, sp_stream_t stream) {
    if (B < 0 || T < 0 || T_pad < T) return set_error(SP_ERR_INVALID_ARG, "sp_pad_mask: bad args");
    if (T_pad == 0 || (user_mask && B == 0)) return SP_OK;  // empty masks may carry null pointers
    if (!mask_out) return set_error(SP_ERR_INVALID_ARG, "sp_pad_mask: mask_out is NULL");
    cudaStream_t st = (cudaStream_t)stream;
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    if (!user_mask) {
        int grid = (T_pad + 255) / 256;
        if (grid > di.num_sms * 4) grid = di.num_sms * 4;
        pad_mask_key_kernel<<<grid, 256, 0, st>>>(mask_out, T, T_pad);
        return check_launch("sp_pad_mask(key)");
    }
    if (B == 0) return SP_OK;
    uint64_t rows = (uint64_t)B * T_pad;
    if (rows > 0x7fffffffull) return set_error(SP_ERR_INVALID_ARG, "sp_pad_mask: too large");
    uint64_t want = (rows + 7) / 8;
    unsigned grid = (unsigned)(want < (uint64_t)di.num_sms * 8 ? want : (uint64_t)di.num_sms * 8);
    pad_mask_user_kernel<<<grid, 256, 0, st>>>(user_mask, mask_out, B, T, T_pad);
    return check_launch("sp_pad_mask(user)");
}

int sp_tile(const void *x_pad, void *const *shards, int W, int B, int T_pad, int64_t row_bytes,
            sp_stream_t stream) {
    if (W < 1 || W > SP_MAX_RANKS || B < 0 || T_pad < 0 || row_bytes < 0 || !shards)
        return set_error(SP_ERR_INVALID_ARG, "sp_tile: bad args");
    if (T_pad % W != 0)
        return set_error(SP_ERR_NOT_DIVISIBLE, "total_tokens=%d is not divisible by world_size=%d", T_pad, W);
    TileOp op;
    memset(&op, 0, sizeof(op));
    op.x = (const uint8_t *)x_pad;
    op.B = B;
    op.Tl = T_pad / W;
    op.T_pad = T_pad;
    op.rb = row_bytes;
    uint64_t align = (uint64_t)(uintptr_t)x_pad | (uint64_t)row_bytes;
    const bool any = (int64_t)B * T_pad * row_bytes > 0;
    if (any && !x_pad) return set_error(SP_ERR_INVALID_ARG, "sp_tile: null input");
    for (int r = 0; r < W; r++) {
        if (any && !shards[r]) return set_error(SP_ERR_INVALID_ARG, "sp_tile: null shard %d", r);
        op.shard[r] = (uint8_t *)shards[r];
        align |= (uint64_t)(uintptr_t)shards[r];
    }
    return launch_rows(op, (uint64_t)B * T_pad, row_bytes, vector_width(align), (cudaStream_t)stream, "sp_tile");
}

int sp_optimal_split(int W, int *split_h, int *split_w) {
    if (W < 1 || !split_h || !split_w) return set_error(SP_ERR_INVALID_ARG, "sp_optimal_split: W=%d", W);
    int a = 1;
    for (int d = 1; (int64_t)d * d <= W; d++)
        if (W % d == 0) a = d;
    *split_h = a;
    *split_w = W / a;
    return SP_OK;
}

int sp_tile_2d(const void *x, void *const *shards, int B, int F, int Hg, int Wg, int split_h, int split_w,
               int64_t row_bytes, sp_stream_t stream) {
    return launch_split_2d<false>(x, (const void *const *)shards, B, F, Hg, Wg, split_h, split_w, row_bytes,
                                  (cudaStream_t)stream, "sp_tile_2d");
}

int sp_gather_2d(const void *const *shards, void *out, int B, int F, int Hg, int Wg, int split_h, int split_w,
                 int64_t row_bytes, sp_stream_t stream) {
    return launch_split_2d<true>(out, shards, B, F, Hg, Wg, split_h, split_w, row_bytes, (cudaStream_t)stream,
                                 "sp_gather_2d");
}

int sp_gather_output(const void *const *shards, void *out, int W, int B, int Tl, int T_out,
                     int64_t row_bytes, sp_stream_t stream) {
    if (W < 1 || W > SP_MAX_RANKS || B < 0 || Tl < 0 || T_out < 0 || row_bytes < 0 || !shards)
        return set_error(SP_ERR_INVALID_ARG, "sp_gather_output: bad args");
    if ((int64_t)T_out > (int64_t)W * Tl)
        return set_error(SP_ERR_INVALID_ARG, "sp_gather_output: T_out=%d > W*Tl=%d", T_out, W * Tl);
    GatherOutOp op;
    memset(&op, 0, sizeof(op));
    op.y = (uint8_t *)out;
    op.Tl = Tl;
    op.T_out = T_out;
    op.rb = row_bytes;
    const bool any = (int64_t)B * T_out * row_bytes > 0;
    if (any && !out) return set_error(SP_ERR_INVALID_ARG, "sp_gather_output: null output");
    uint64_t align = (uint64_t)(uintptr_t)out | (uint64_t)row_bytes;
    for (int r = 0; r < W; r++) {
        const bool used = (int64_t)r * Tl < T_out;
        if (any && used && !shards[r]) return set_error(SP_ERR_INVALID_ARG, "sp_gather_output: null shard %d", r);
        op.shard[r] = (const uint8_t *)shards[r];
        align |= (uint64_t)(uintptr_t)shards[r];
    }
    return launch_rows(op, (uint64_t)B * T_out, row_bytes, vector_width(align), (cudaStream_t)stream,
                       "sp_gather_output");
}

int sp_send_recv_heads(const void *const *shards, void *const *heads, int W, int B, int Tl, int H,
                       int D, int elt_bytes, void *workspace, sp_stream_t stream) {
    return launch_exchange<false>(shards, heads, W, B, Tl, H, D, elt_bytes, workspace,
                                  (cudaStream_t)stream, "sp_send_recv_heads");
}

int sp_gather_heads(const void *const *heads, void *const *shards, int W, int B, int Tl, int H,
                    int D, int elt_bytes, void *workspace, sp_stream_t stream) {
    return launch_exchange<true>(heads, shards, W, B, Tl, H, D, elt_bytes, workspace,
                                 (cudaStream_t)stream, "sp_gather_heads");
}

int sp_send_recv_heads_noalloc(const void *const *shards, void *const *heads, int W, int B, int Tl, int H,
                               int D, int elt_bytes, int *status_out, sp_stream_t stream) {
    if (W < 1 || W > SP_MAX_RANKS)
        return set_error(SP_ERR_INVALID_ARG,
                         "sp_send_recv_heads_noalloc: W=%d, but the static scratch holds counters for at most %d ranks",
                         W, SP_MAX_RANKS);
    void *ws = nullptr;
    int rc = noalloc_scratch(&ws);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    const char *what = "sp_send_recv_heads_noalloc";
    ExchangeParams p;
    int V = 16;
    // every argument is checked before the shared array is touched: a
    // rejected call leaves it as the previous call left it
    rc = prepare_exchange(shards, heads, W, B, Tl, H, D, elt_bytes, ws, what, p, V);
    if (rc) return rc;
    // the ticket and the counters must start at zero (the previous call's
    // last CTA reset them; cleared again in case that call never ran to its
    // end).  The status word is kept: it holds the first device error since
    // the last read, which a call with status_out reports and resets.
    SP_CUDA_CHECK(cudaMemsetAsync((uint8_t *)ws + offsetof(WorkspaceHeader, ticket), 0,
                                  offsetof(WorkspaceHeader, observed) - offsetof(WorkspaceHeader, ticket), st));
    rc = run_exchange<false>(p, V, st, what);
    if (rc) return rc;
    if (status_out) {
        int s = 0;
        SP_CUDA_CHECK(cudaMemcpyAsync(&s, ws, sizeof(int), cudaMemcpyDeviceToHost, st));
        SP_CUDA_CHECK(cudaStreamSynchronize(st));
        *status_out = s;
        SP_CUDA_CHECK(cudaMemsetAsync(ws, 0, sizeof(int), st));
    }
    return SP_OK;
}

int sp_pad_send_heads(const void *x, void *const *heads, int W, int B, int T, int T_pad, int H, int D,
                      int elt_bytes, void *workspace, sp_stream_t stream) {
    return launch_exchange_fused<false>(const_cast<void *>(x), heads, W, B, T_pad, T, H, D, elt_bytes, workspace,
                                        (cudaStream_t)stream, "sp_pad_send_heads");
}

int sp_gather_heads_output(const void *const *heads, void *out, int W, int B, int T_pad, int T_out, int H, int D,
                           int elt_bytes, void *workspace, sp_stream_t stream) {
    return launch_exchange_fused<true>(out, const_cast<void *const *>(heads), W, B, T_pad, T_out, H, D, elt_bytes,
                                       workspace, (cudaStream_t)stream, "sp_gather_heads_output");
}

int sp_workspace_status(void *workspace, int *status, int *counts, int *n_launches, int clear,
                        sp_stream_t stream) {
    if (!workspace || !status) return set_error(SP_ERR_INVALID_ARG, "sp_workspace_status: null");
    cudaStream_t st = (cudaStream_t)stream;
    WorkspaceHeader h;
    SP_CUDA_CHECK(cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st));
    SP_CUDA_CHECK(cudaStreamSynchronize(st));
    *status = h.status;
    if (counts)
        for (int r = 0; r < SP_MAX_RANKS; r++) counts[r] = h.observed[r];
    if (n_launches) *n_launches = h.launches;
    if (clear) {
        SP_CUDA_CHECK(cudaMemsetAsync(workspace, 0, sizeof(int), st));
        SP_CUDA_CHECK(cudaStreamSynchronize(st));
    }
    return SP_OK;
}

}  // extern "C"
