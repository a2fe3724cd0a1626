// CUDA-core attention for the shapes the tensor-core kernel does not cover:
// fp32 inputs (where tensor-core TF32 would miss a 1e-4 bound) and bf16 with
// a head dim other than 64 or 128.
//
// Source: "LTX-2 序列并行拆解", section 换头: after the exchange every rank
// computes attention on its local heads over all tokens.
//
// One warp owns one query row (rank, batch, head, query).  Lane j holds the
// query and output elements d = j, j+32, ...; keys are visited in increasing
// order with an online softmax in fp32, so the result does not depend on the
// padding or sharding of the key sequence: masked keys are skipped outright.
#include <cuda_bf16.h>

#include "sp_attn.cuh"

namespace sp {

template <typename T>
__device__ __forceinline__ float ld_f(const T *p);
template <>
__device__ __forceinline__ float ld_f<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ void st_f(T *p, float v);
template <>
__device__ __forceinline__ void st_f<float>(float *p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_f<__nv_bfloat16>(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T, int NJ>
__global__ void __launch_bounds__(256) attn_simt_kernel(AttnArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nrows = (int64_t)a.W * a.B * a.Hl * a.Tq;
    if (row >= nrows) return;
    // row -> (r, b, h, q), q fastest
    int64_t t = row;
    const int q = (int)(t % a.Tq); t /= a.Tq;
    const int h = (int)(t % a.Hl); t /= a.Hl;
    const int b = (int)(t % a.B); t /= a.B;
    const int r = (int)t;

    const T *Q = (const T *)a.q[r] + b * a.qs[0] + (int64_t)q * a.qs[1] + h * a.qs[2];
    const T *K = (const T *)a.k[r] + b * a.ks[0] + h * a.ks[2];
    const T *V = (const T *)a.v[r] + b * a.ks[0] + h * a.ks[2];
    T *O = (T *)a.o[r] + b * a.os[0] + (int64_t)q * a.os[1] + h * a.os[2];

    float qv[NJ], acc[NJ];
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        const int d = lane + 32 * j;
        qv[j] = d < a.D ? ld_f<T>(Q + d) : 0.f;
        acc[j] = 0.f;
    }
    const uint8_t *mrow = nullptr;
    if (a.mask_kind == SP_MASK_KEY) mrow = a.mask;
    else if (a.mask_kind == SP_MASK_FULL) mrow = a.mask + ((int64_t)b * a.Tq + q) * a.Tk;

    float m = -INFINITY, l = 0.f;
    for (int k = 0; k < a.Tk; k++) {
        if (mrow && mrow[k] == 0) continue;  // uniform across the warp
        const T *kr = K + (int64_t)k * a.ks[1];
        float dot = 0.f;
#pragma unroll
        for (int j = 0; j < NJ; j++) {
            const int d = lane + 32 * j;
            if (d < a.D) dot = fmaf(qv[j], ld_f<T>(kr + d), dot);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const float s = dot * a.scale;
        const float m_new = fmaxf(m, s);
        const float corr = expf(m - m_new);  // m = -inf on the first visible key -> 0
        const float p = expf(s - m_new);
        l = l * corr + p;
        const T *vr = V + (int64_t)k * a.ks[1];
#pragma unroll
        for (int j = 0; j < NJ; j++) {
            const int d = lane + 32 * j;
            const float vv = d < a.D ? ld_f<T>(vr + d) : 0.f;
            acc[j] = fmaf(p, vv, acc[j] * corr);
        }
        m = m_new;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        const int d = lane + 32 * j;
        if (d < a.D) st_f<T>(O + d, acc[j] * inv);
    }
}

template <typename T>
static void launch_simt_t(const AttnArgs &a, cudaStream_t st) {
    const int64_t rows = (int64_t)a.W * a.B * a.Hl * a.Tq;
    const int64_t blocks = (rows * 32 + 255) / 256;
    const int nj = (a.D + 31) / 32;
    switch (nj) {
        case 1: attn_simt_kernel<T, 1><<<(unsigned)blocks, 256, 0, st>>>(a); break;
        case 2: attn_simt_kernel<T, 2><<<(unsigned)blocks, 256, 0, st>>>(a); break;
        case 3: attn_simt_kernel<T, 3><<<(unsigned)blocks, 256, 0, st>>>(a); break;
        case 4: attn_simt_kernel<T, 4><<<(unsigned)blocks, 256, 0, st>>>(a); break;
        case 5: attn_simt_kernel<T, 5><<<(unsigned)blocks, 256, 0, st>>>(a); break;
        case 6: attn_simt_kernel<T, 6><<<(unsigned)blocks, 256, 0, st>>>(a); break;
        case 7: attn_simt_kernel<T, 7><<<(unsigned)blocks, 256, 0, st>>>(a); break;
        default: attn_simt_kernel<T, 8><<<(unsigned)blocks, 256, 0, st>>>(a); break;
    }
}

int launch_attn_simt(const AttnArgs &a, cudaStream_t st) {
    const int64_t rows = (int64_t)a.W * a.B * a.Hl * a.Tq;
    if (rows == 0) return SP_OK;
    if (rows * 32 / 256 + 1 > 0x7fffffffll) return set_error(SP_ERR_INVALID_ARG, "sp_attention: too many rows");
    if (a.dtype == SP_F32) launch_simt_t<float>(a, st);
    else launch_simt_t<__nv_bfloat16>(a, st);
    return check_launch("sp_attention(simt)");
}

}  // namespace sp
