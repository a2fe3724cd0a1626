// Tensor-core flash attention for sm_103a: tcgen05.mma with TMEM accumulators,
// operands staged by TMA, online softmax, key masking and the pad-row rule
// fused in; one launch covers every virtual rank x batch x local head x query
// tile.
//
// Source: "LTX-2 序列并行拆解", section 换头 (after send_recv_heads each rank
// holds all tokens x H/W heads and computes attention on them in place) and
// section 补齐 (key-only padding mask / extended user mask; pad query rows see
// the valid keys).  The pages name no attention kernel; this design is new.
//
// CTA = one (rank, batch, head) and a PAIR of 128-row query tiles (Q0, Q1)
// sharing every K/V tile, so the tensor core always has one tile's GEMMs
// queued while the other tile's softmax runs.  320 threads, 1 CTA per SM:
//   warps 0-3  softmax for Q0 (thread = query row, TMEM lanes 0..127)
//   warps 4-7  softmax for Q1
//   warp  8    TMA producer (Q once; K and V tiles through one shared ring of
//              NSLOT slots, loaded in the order K0 V0 K1 V1 ...)
//   warp  9    TMEM allocator + single-thread MMA issuer
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [384,384+D).
// P (bf16) overwrites the first 64 columns of its S buffer and feeds the PV
// GEMM straight from TMEM (A operand in TMEM, V from shared memory).
// The softmax takes each row's maximum from the TMEM load of S itself
// (tcgen05.ld.red); only a tile with hidden keys recomputes it over the
// visible ones.
// Per KV tile j the MMA issue order is
//   PV0(j) QK0(j+1) PV1(j) QK1(j+1)
// so S_i(j+1) is written only after PV_i(j) has consumed P_i(j) (tcgen05
// operations of one thread execute in issue order), and the commit that
// signals S_i(j+1) also proves O_i holds PV_i(j) -- the softmax warps may
// rescale O_i right away.  Rescaling is lazy: the running max moves only when
// a tile's max exceeds it by more than 8 (log2 units), which keeps every
// probability <= 2^8 and makes O rescales rare.
//
// Work decomposition (plan_split): a work item is one (rank, batch, head,
// query pair).  Short query sequences (fewer items than SMs) cut every item
// into key pieces, and a last, partial wave of items is cut likewise; the
// pieces' fp32 partials are merged by LSE in attn_merge_kernel.
// Operands are either each rank's tensors or, for the exchange fused into
// the attention, the source ranks' token shards (Tiling): every shard's whole
// 128-row tiles, and its leftover block when that holds at least half a tile,
// come by TMA from the shard; smaller leftover blocks are gathered into tiles
// that the producer warp copies row by row into the same swizzled layout.
//
// Every mbarrier wait is bounded (%globaltimer); on timeout the CTA records
// SP_ERR_TIMEOUT, every role stops, in-flight copies and MMAs are drained
// (again with a bound) and TMEM is freed before the CTA exits.
#include <atomic>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include "sp_attn.cuh"

namespace sp {
namespace tc {

constexpr int kThreads = 320;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr float kRescaleThreshold = 8.0f;      // log2 units

template <int D>
struct Cfg {
    static constexpr int DB = D / 64;             // 128-byte swizzle blocks per row
    static constexpr int TILE = 128 * D * 2;      // bytes of a 128-row bf16 tile
    static constexpr int NSLOT = (D == 64) ? 10 : 5;  // K/V ring slots (2.5 tiles of each ahead at D=128)
    static constexpr int Q_OFF = 0;
    static constexpr int R_OFF = 2 * TILE;
    static constexpr int BYTES = R_OFF + NSLOT * TILE;
    static constexpr int SMEM_ALLOC = BYTES + 1024;  // + slack to align the base to 1024
};

// How the 128-row tiles of one operand map onto its memory.  A per-rank
// tensor (sharded == 0): tile j is rows [128 j, 128 j + 128).  W source token
// shards (sharded != 0): global token g lives in shard g / Tl at row g % Tl,
// and shard s holds rows[s] real rows.  The tiles are, in this order:
//   - every shard's whole 128-row tiles, in shard order (shard s owns tiles
//     [full0[s], full0[s+1]));
//   - "partial" tiles: one per shard whose leftover block (rows[s] % 128
//     rows after its whole tiles) holds at least kPartialMin rows, loaded by
//     TMA from the shard like a whole tile, the rows past the shard's end
//     reading as zeros and masked off (shards part[0 .. npart));
//   - "gathered" tiles from tile g0 = full0[W] + npart on: the smaller
//     leftover blocks, packed in shard order (shard s's are gathered slots
//     [tail0[s], tail0[s+1])) and copied row by row; slots past tail0[W]
//     hold no token.
// With Tl a multiple of 128 (and only the last shard short) the tiles are
// exactly global rows [128 j, 128 j + 128), the order of the exchanged layout.
constexpr int kPartialMin = 64;
struct Tiling {
    int sharded;
    int Tl;
    int npart, g0;
    int rows[SP_MAX_RANKS];
    int part[SP_MAX_RANKS];
    int full0[SP_MAX_RANKS + 1];
    int tail0[SP_MAX_RANKS + 1];
};

struct alignas(128) TcParams {
    CUtensorMap tq[SP_MAX_RANKS], tk[SP_MAX_RANKS], tv[SP_MAX_RANKS], to[SP_MAX_RANKS];
    int W, B, Tq, Tk, Hl;
    int n_qpairs, n_kv, n_split, kv_per_split;
    int n_full;  // SPLIT launches: work items [0, n_full) run whole, the rest in n_split key pieces
    // Tilings of Q/O and of K/V.  A sharded operand's maps are per source
    // token shard, addressed with head r * Hl + h; tail tiles are copied by
    // the producer warp from the raw pointers below (strides in elements).
    Tiling qtl, ktl;
    const uint8_t *qptr[SP_MAX_RANKS], *kptr[SP_MAX_RANKS], *vptr[SP_MAX_RANKS];
    uint8_t *optr[SP_MAX_RANKS];
    int64_t qs[3], ks[3], os[3];
    float scale_log2;
    int mask_kind, mask_vec4;
    const uint8_t *mask;
    float *part_o;    // split partials [item][split][256][D]
    float *part_lse;  // [item][split][256], log2 domain
    int *status;
    const int *kv_stall;  // workspace test hook (see SP_WORKSPACE_KV_STALL_OFFSET)
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// Raises the transaction count of the current phase without an arrival.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void st_shared_zero16(uint32_t dst) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u));
}
// 16-byte global -> shared copy; src_bytes = 0 writes 16 zero bytes and reads nothing.
// (No memory clobber: nothing in C++ reads the destination before the wait
// below, which has one; so operands loaded before the loop stay in registers.)
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// Slow path of wait_bounded: poll with a %globaltimer bound.
__device__ __noinline__ bool wait_slow(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *status) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 32; i++)
            if (mbar_try_wait(a, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kTimeoutNs) {
            *abort_flag = 1;
            atomicCAS(status, 0, SP_ERR_TIMEOUT);
            return false;
        }
    }
}
// Bounded wait: false when this CTA has aborted or the wait timed out (which
// aborts the CTA and records SP_ERR_TIMEOUT).  The first try is inline.
__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                             int *status) {
    if (mbar_try_wait(smem_u32(bar), parity)) return true;
    return wait_slow(bar, parity, abort_flag, status);
}
// Drain wait (teardown after an abort): bounded, ignores the abort flag.
__device__ __noinline__ void wait_drain(uint64_t *bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(a, parity))
        if (globaltimer() - t0 > kTimeoutNs) return;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint64_t *bar, const CUtensorMap *m, uint32_t dst, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *m, uint32_t src, int c0, int c1, int c2,
                                             int c3) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Named barrier that also ANDs a predicate over its participants.
__device__ __forceinline__ bool named_bar_and(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D(tmem) (+)= A(smem) * B(smem)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, A K-major,
// B K-major (b_mn = false) or MN-major (b_mn = true), shape M x N.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn) {
    return (1u << 4)                        // D format: f32
           | (1u << 7)                      // A format: bf16
           | (1u << 10)                     // B format: bf16
           | ((b_mn ? 1u : 0u) << 16)       // B major-ness
           | ((uint32_t)(N >> 3) << 17)     // N / 8
           | ((uint32_t)(M >> 4) << 24);    // M / 16
}
// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;  // SWIZZLE_128B
    return d;
}

// TMEM loads/stores; the load wrappers include the wait so the compiler never
// reads the destination registers early.
// 128 columns of this warp's 32 TMEM lanes (one row per thread), and each
// thread's maximum over its 128 values, reduced as they leave TMEM
// (tcgen05.ld.red, sm_103a).
__device__ __forceinline__ void tmem_ld_max_x128(uint32_t taddr, uint32_t (&r)[128], float &mx) {
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x128.max.f32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, %128, [%129];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127]), "=f"(mx)
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_st_x64(uint32_t taddr, const uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};\n"
        :
        : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
        : "memory");
}

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n"
        :
        : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}


__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// Two fp32 lanes in one 64-bit register, for the packed f32x2 arithmetic.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ uint64_t f2_pack_u(uint32_t lo, uint32_t hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t nibble_of(uint32_t v) {
    return ((v & 0x000000ffu) ? 1u : 0u) | ((v & 0x0000ff00u) ? 2u : 0u) | ((v & 0x00ff0000u) ? 4u : 0u) |
           ((v & 0xff000000u) ? 8u : 0u);
}
// Mask bytes of keys [k, k+4) of one mask row, as one word (bounds-checked:
// a key past Tk reads as masked).  nibble_of turns it into visibility bits.
__device__ __forceinline__ uint32_t mask_raw4(const uint8_t *row, int k, int Tk, bool vec4) {
    if (vec4 && k + 3 < Tk) return *reinterpret_cast<const uint32_t *>(row + k);
    uint32_t v = 0;
#pragma unroll
    for (int e = 0; e < 4; e++)
        if (k + e < Tk && row[k + e]) v |= 0xffu << (8 * e);
    return v;
}
// Visibility bits of keys [k, k+4) of one mask row.
__device__ __forceinline__ uint32_t mask_nibble(const uint8_t *row, int k, int Tk, bool vec4) {
    return nibble_of(mask_raw4(row, k, Tk, vec4));
}
// The 128 bits of a key tile from each lane's nibble (lane L holds keys
// 4L .. 4L+3), gathered across the warp.
__device__ __forceinline__ void nibbles_to_words(uint32_t nib, int lane, uint32_t w[4]) {
    uint32_t word = nib << (4 * (lane & 7));
    word |= __shfl_xor_sync(0xffffffffu, word, 1);
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    word |= __shfl_xor_sync(0xffffffffu, word, 4);
    w[0] = __shfl_sync(0xffffffffu, word, 0);
    w[1] = __shfl_sync(0xffffffffu, word, 8);
    w[2] = __shfl_sync(0xffffffffu, word, 16);
    w[3] = __shfl_sync(0xffffffffu, word, 24);
}

// 128 visibility bits (4 words) of keys [key0, key0+128) for this thread's row.
__device__ __forceinline__ void mask_words(const TcParams &p, int b, int q_row, int key0, int lane,
                                           uint32_t w[4]) {
    if (p.mask_kind == SP_MASK_KEY) {
        // warp-cooperative: lane covers keys key0 + 4*lane .. +3
        nibbles_to_words(mask_nibble(p.mask, key0 + 4 * lane, p.Tk, p.mask_vec4), lane, w);
        return;
    }
    if (p.mask_kind == SP_MASK_FULL && q_row < p.Tq) {
        const uint8_t *row = p.mask + ((int64_t)b * p.Tq + q_row) * p.Tk;
#pragma unroll
        for (int g = 0; g < 4; g++) {
            uint32_t word = 0;
#pragma unroll
            for (int n = 0; n < 8; n++) word |= mask_nibble(row, key0 + 32 * g + 4 * n, p.Tk, p.mask_vec4) << (4 * n);
            w[g] = word;
        }
        return;
    }
    // no mask (or a query row past Tq): keys < Tk are visible
#pragma unroll
    for (int g = 0; g < 4; g++) {
        const int n = p.Tk - (key0 + 32 * g);
        w[g] = n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
    }
}

// Tile j of a sharded operand when TMA loads it (a whole or a partial tile):
// its shard s, first row and the number of its rows that hold tokens; false
// for a gathered tile (or past the last tile).
__device__ __forceinline__ bool tiling_box(const Tiling &t, int W, int j, int &s, int &row, int &nvalid) {
    if (j < t.full0[W]) {
        int q = 0;
        while (q + 1 < W && j >= t.full0[q + 1]) q++;
        s = q;
        row = (j - t.full0[q]) * 128;
        nvalid = 128;
        return true;
    }
    const int k = j - t.full0[W];
    if (k >= t.npart) return false;
    s = t.part[k];
    row = (t.full0[s + 1] - t.full0[s]) * 128;
    nvalid = t.rows[s] - row;
    return true;
}
// Gathered slot idx: its shard s and row; false past the last gathered row.
__device__ __forceinline__ bool tiling_tail(const Tiling &t, int W, int idx, int &s, int &row) {
    if (idx < 0 || idx >= t.tail0[W]) return false;
    int q = 0;
    while (q + 1 < W && idx >= t.tail0[q + 1]) q++;
    s = q;
    row = (t.full0[q + 1] - t.full0[q]) * 128 + (idx - t.tail0[q]);
    return true;
}
// Where tile j of rank r's local head h comes from when TMA can load it:
// the rank's own tensor (map r, head h, rows [128 j, 128 j + 128)) or a
// whole or partial tile of source shard s (map s, head r * Hl + h).  False
// for a gathered tile, which the producer warp assembles row by row.
__device__ __forceinline__ bool tile_src(const Tiling &t, int W, int j, int r, int h, int Hl, int &map, int &head,
                                         int &row) {
    if (!t.sharded) {
        map = r;
        head = h;
        row = j * 128;
        return true;
    }
    head = r * Hl + h;
    int nvalid;
    return tiling_box(t, W, j, map, row, nvalid);
}
// Global token of row e of tile j, or -1 when the slot holds none.
__device__ __forceinline__ int tile_token(const Tiling &t, int W, int j, int e) {
    if (!t.sharded) return j * 128 + e;
    int s, row, nvalid;
    if (tiling_box(t, W, j, s, row, nvalid)) return e < nvalid ? s * t.Tl + row + e : -1;
    if (tiling_tail(t, W, (j - t.g0) * 128 + e, s, row)) return s * t.Tl + row;
    return -1;
}

// Gathered tile tt of a sharded operand into the 128-byte-swizzled tile at
// shared address dst (the layout a TMA box writes: 64-column blocks 16 KB
// apart, row e at e * 128, 16-byte chunk c at (c ^ (e & 7)) * 16), by all 32
// lanes of the calling warp with 16-byte copies.  base: the W shards; st:
// batch, token, head strides (elements).  Each lane walks its rows (every
// RPI-th slot) with a running source pointer, recomputed only where the walk
// crosses into the next shard.  Slots past the last gathered row are left as
// they are, or zeroed when zero_empty: an empty K row is masked whatever it
// holds, and an empty Q row yields an output row that is never stored, but an
// empty V row is multiplied by P = 0 and must not hold non-finite bits, which
// only a slot this CTA has not filled before can.
template <int D>
__device__ __forceinline__ void fill_tail(uint32_t dst, const Tiling &t, int W, int tt, const uint8_t *const *base,
                                          const int64_t *st, int b, int head, int lane, bool zero_empty) {
    constexpr int CPR = D / 8;     // 16-byte chunks per row
    constexpr int RPI = 32 / CPR;  // rows per pass of the warp
    const int c = lane % CPR;
    const int64_t row_stride = st[1] * 2;
    const int64_t off = ((int64_t)b * st[0] + (int64_t)head * st[2]) * 2 + c * 16;
    const int nvalid = min(max(t.tail0[W] - tt * 128, 0), 128);
    int e = lane / CPR, idx = tt * 128 + e;
    if (e < nvalid) {
        int s = 0;
        while (s + 1 < W && idx >= t.tail0[s + 1]) s++;
        int end = t.tail0[s + 1];
        const uint8_t *src =
            base[s] + off + ((int64_t)(t.full0[s + 1] - t.full0[s]) * 128 + (idx - t.tail0[s])) * row_stride;
        for (; e < nvalid; e += RPI, idx += RPI, src += RPI * row_stride) {
            while (idx >= end && s + 1 < W) {
                s++;
                end = t.tail0[s + 1];
                src = base[s] + off +
                      ((int64_t)(t.full0[s + 1] - t.full0[s]) * 128 + (idx - t.tail0[s])) * row_stride;
            }
            const uint32_t d = dst + (uint32_t)((c >> 3) * 16384 + e * 128 + (((c & 7) ^ (e & 7)) << 4));
            cp_async_16(d, src, 16u);
        }
    }
    if (zero_empty)
        for (; e < 128; e += RPI)
            st_shared_zero16(dst + (uint32_t)((c >> 3) * 16384 + e * 128 + (((c & 7) ^ (e & 7)) << 4)));
    cp_async_wait_all();
    fence_proxy_async_smem();  // the tensor core (async proxy) reads what these copies wrote
}

// Visibility bits of tail key tile tt for this thread's query row (global
// token q_row, or >= Tq for a slot without a query): slots past the last
// leftover row are never visible.
__device__ __forceinline__ void tail_words(const TcParams &p, int b, int q_row, int tt, int lane, uint32_t w[4]) {
    const Tiling &t = p.ktl;
    const int nvalid = min(max(t.tail0[p.W] - tt * 128, 0), 128);
    if (p.mask_kind == SP_MASK_KEY) {
        // warp-cooperative: lane covers slots 4*lane .. +3
        uint32_t nib = 0;
#pragma unroll
        for (int e = 0; e < 4; e++) {
            int s, row;
            if (tiling_tail(t, p.W, tt * 128 + 4 * lane + e, s, row) && p.mask[s * t.Tl + row]) nib |= 1u << e;
        }
        nibbles_to_words(nib, lane, w);
        return;
    }
    if (p.mask_kind == SP_MASK_FULL && q_row < p.Tq) {
        const uint8_t *mrow = p.mask + ((int64_t)b * p.Tq + q_row) * p.Tk;
        for (int g = 0; g < 4; g++) w[g] = 0u;
        for (int e = 0; e < nvalid; e++) {
            int s, row;
            tiling_tail(t, p.W, tt * 128 + e, s, row);
            if (mrow[s * t.Tl + row]) w[e >> 5] |= 1u << (e & 31);
        }
        return;
    }
#pragma unroll
    for (int g = 0; g < 4; g++) {
        const int n = nvalid - 32 * g;
        w[g] = n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
    }
}

// Visibility bits of key tile j (any tiling) for this thread's query row.
__device__ __forceinline__ void key_words(const TcParams &p, int b, int q_row, int j, int lane, uint32_t w[4]) {
    int s, row;
    int nvalid;
    if (!p.ktl.sharded) {
        mask_words(p, b, q_row, j * 128, lane, w);
    } else if (p.mask_kind == SP_MASK_NONE && j < p.ktl.full0[p.W]) {
        w[0] = w[1] = w[2] = w[3] = 0xffffffffu;  // a whole tile of real keys
    } else if (tiling_box(p.ktl, p.W, j, s, row, nvalid)) {
        mask_words(p, b, q_row, s * p.ktl.Tl + row, lane, w);  // consecutive tokens of shard s
        if (nvalid < 128) {  // a partial tile: its rows past the shard's end hold no key
#pragma unroll
            for (int g = 0; g < 4; g++) {
                const int n = nvalid - 32 * g;
                w[g] &= n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
            }
        }
    } else {
        tail_words(p, b, q_row, j - p.ktl.g0, lane, w);
    }
}

// key_words out of line, for the softmax loop of the sharded instance: there
// the usual tile is a whole tile of unmasked keys, decided by one comparison,
// and the rare others (partial and gathered tiles, masks) take this call, so
// the loop's own code stays as small as the unsharded instance's.
__device__ __noinline__ uint4 key_words_call(const TcParams &p, int b, int q_row, int j, int lane) {
    uint32_t w[4];
    key_words(p, b, q_row, j, lane, w);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// ------------------------------------------------------------------ kernel
// TILED: some operand is a set of token shards (see Tiling); otherwise every
// operand is a per-rank tensor and the tile arithmetic is the plain one.
template <int D, bool SPLIT, bool TILED>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ TcParams p) {
    using C = Cfg<D>;
    constexpr int NSLOT = C::NSLOT;  // ring slots
    constexpr int SLOT = C::TILE;    // bytes per slot
    extern __shared__ uint8_t dsm_raw[];
    // Ring slots are freed by release events, one tcgen05.commit each: event
    // 0 (after QK1(0)) frees K(0); event e >= 1 (after QK1(e), issued in step
    // e-1, which also orders PV1(e-1) before it) frees V(e-1) and K(e), the
    // loads 2e-1 and 2e.  So load m is free after event ceil(m / 2).  Events
    // go round NREL barriers: while the producer waits for event e before
    // its load n = m + NSLOT, at most n - 1 <= 2e + NSLOT - 1 loads exist, and
    // event e + NREL needs load 2(e + NREL) > that, so a barrier never runs a
    // whole phase past the one its waiter expects.
    // No tcgen05.commit signals them: the S1(j) commit already marks event j's
    // completion point, so the first lane of tile 1's first softmax warp,
    // which waits for it anyway, relays event j with a plain arrive: at the
    // end of its iteration j, or, in the sharded instance, as soon as S1(j)
    // is in registers (each place measured fastest for its instance).
    constexpr int NREL = NSLOT / 2 + 1;
    __shared__ __align__(8) uint64_t bar_q, bar_full[NSLOT], bar_rel[NREL];
    __shared__ __align__(8) uint64_t bar_sf[2], bar_pf[2], bar_of[2], bar_drain;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t raw = smem_u32(dsm_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *const sgen = dsm_raw + (sbase - raw);

    // work item: blockIdx.x -> (rank, batch, head, key split, query pair), query pair
    // fastest
    //
    // SPLIT launches: CTAs [0, n_full) take work items [0, n_full) whole; each
    // later item (the ones that would otherwise form a last, partial wave, or
    // every item of a short query sequence) is cut into n_split key ranges
    // whose partial results attn_merge_kernel combines.  `piece` < 0: whole.
    int bid = blockIdx.x;
    int qp, piece = -1;
    int64_t witem = 0;  // work item, (((r * B + b) * Hl + h) * n_qpairs + qp)
    int kv0, kv1;
    if (!SPLIT) {
        qp = bid % p.n_qpairs;
        bid /= p.n_qpairs;
        // (n_split is 1 here; the key range is still derived from the grid,
        // which keeps this instance's code as it measured fastest)
        const int split = bid % p.n_split;
        bid /= p.n_split;
        kv0 = split * p.kv_per_split;
        kv1 = min(p.n_kv, kv0 + p.kv_per_split);
    } else {
        if (bid < p.n_full) {
            witem = bid;
        } else {
            const int u = bid - p.n_full;
            witem = p.n_full + u / p.n_split;
            piece = u % p.n_split;
        }
        qp = (int)(witem % p.n_qpairs);
        bid = (int)(witem / p.n_qpairs);
        kv0 = piece < 0 ? 0 : piece * p.kv_per_split;
        kv1 = piece < 0 ? p.n_kv : min(p.n_kv, kv0 + p.kv_per_split);
    }
    const int h = bid % p.Hl;
    bid /= p.Hl;
    const int b = bid % p.B;
    const int r = bid / p.B;
    const int nkv = max(0, kv1 - kv0);
    // CTAs of one head run in step; starting each query pair at a different key
    // tile spreads their concurrent K/V reads over L2 instead of all CTAs asking
    // for the same tile at once.  Softmax is order-free, so only rounding moves.
    const int rot = nkv > 0 ? (int)(((unsigned)(qp >> 1) * 7u) % (unsigned)nkv) : 0;
    auto key_tile = [&](int jj) { int t = jj + rot; return kv0 + (t >= nkv ? t - nkv : t); };

    // a split launch is followed by attn_merge_kernel, launched as its
    // programmatic dependent: let its CTAs be scheduled once every CTA of this
    // grid is running (they wait for this grid's completion before reading)
    if (SPLIT && threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        mbar_init(&bar_q, 1);
        for (int s = 0; s < NSLOT; s++) {
            mbar_init(&bar_full[s], 1);
        }
        for (int s = 0; s < NREL; s++) {
            mbar_init(&bar_rel[s], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&bar_sf[i], 1);
            mbar_init(&bar_pf[i], 128);
            mbar_init(&bar_of[i], 1);
        }
        mbar_init(&bar_drain, 1);
        abort_sh = 0;
        fence_mbarrier_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(&tmem_base_sh), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base_sh;
    volatile int *abort_flag = &abort_sh;

    if (warp == 8) {
        // ---------------------------------------------------------- TMA producer
        if (!TILED && lane == 0 && nkv > 0) {
            prefetch_tmap(&p.tq[r]);
            prefetch_tmap(&p.tk[r]);
            prefetch_tmap(&p.tv[r]);
            mbar_arrive_expect_tx(&bar_q, 2 * C::TILE);
            for (int i = 0; i < 2; i++) {
                for (int db = 0; db < C::DB; db++) {
                    const uint32_t dst = sbase + C::Q_OFF + i * C::TILE + db * 16384;
                    tma_load_4d(&bar_q, &p.tq[r], dst, db * 64, h, qp * 256 + i * 128, b);
                }
            }
            // load n: K of key tile n/2 (n even) or V (n odd) into slot n % NSLOT
            const int stall = *p.kv_stall;  // 0 in normal use
            const int nloads = stall > 0 ? min(2 * nkv, stall - 1) : 2 * nkv;
            int n = 0;
            for (; n < nloads; n++) {
                const int slot = n % NSLOT;
                const int use = n / NSLOT;
                if (use > 0) {  // the slot's previous load (n - NSLOT) has been consumed
                    const int e = (n - NSLOT + 1) >> 1;
                    if (!wait_bounded(&bar_rel[e % NREL], (uint32_t)(e / NREL) & 1u, abort_flag, p.status)) break;
                }
                mbar_arrive_expect_tx(&bar_full[slot], SLOT);
                const CUtensorMap *m = (n & 1) ? &p.tv[r] : &p.tk[r];
                const int krow = key_tile(n >> 1) * 128;
                for (int db = 0; db < C::DB; db++)
                    tma_load_4d(&bar_full[slot], m, sbase + C::R_OFF + slot * C::TILE + db * 16384, db * 64, h, krow,
                                b);
            }
            // Before the CTA may exit, every load it issued has landed: wait
            // for the newest load of every slot (older ones were consumed
            // before their slot was reused).  In a normal run the MMA thread
            // waits for the same phases; after an abort these bounded waits
            // keep the teardown from freeing shared memory under a copy.
            wait_drain(&bar_q, 0);
            for (int slot = 0; slot < NSLOT && slot < n; slot++) {
                const int last = slot + ((n - 1 - slot) / NSLOT) * NSLOT;
                wait_drain(&bar_full[slot], (uint32_t)(last / NSLOT) & 1u);
            }
        } else if (TILED && nkv > 0) {
            // The whole warp runs the loop: lane 0 waits and issues the TMA
            // loads of whole tiles; a tail tile is copied by all 32 lanes and
            // then announced by one plain arrival.
            if (lane < p.W) {
                prefetch_tmap(&p.tq[lane]);
                prefetch_tmap(&p.tk[lane]);
                prefetch_tmap(&p.tv[lane]);
            }
            int qmap[2], qhead[2], qrow[2];
            bool qwhole[2];
            uint32_t qbytes = 0;
            for (int i = 0; i < 2; i++) {
                qwhole[i] = tile_src(p.qtl, p.W, 2 * qp + i, r, h, p.Hl, qmap[i], qhead[i], qrow[i]);
                if (qwhole[i]) qbytes += C::TILE;
            }
            if (lane == 0) {
                if (qbytes) mbar_expect_tx(&bar_q, qbytes);
                for (int i = 0; i < 2; i++)
                    if (qwhole[i])
                        for (int db = 0; db < C::DB; db++)
                            tma_load_4d(&bar_q, &p.tq[qmap[i]], sbase + C::Q_OFF + i * C::TILE + db * 16384, db * 64,
                                        qhead[i], qrow[i], b);
            }
            for (int i = 0; i < 2; i++)
                if (!qwhole[i])
                    fill_tail<D>(sbase + C::Q_OFF + i * C::TILE, p.qtl, p.W, 2 * qp + i - p.qtl.g0, p.qptr,
                                 p.qs, b, qhead[i], lane, false);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_q);
            const int stall = *p.kv_stall;  // 0 in normal use
            const int nloads = stall > 0 ? min(2 * nkv, stall - 1) : 2 * nkv;
            int n = 0;
            for (; n < nloads; n++) {
                const int slot = n % NSLOT;
                const int use = n / NSLOT;
                bool ok = true;
                if (use > 0 && lane == 0)
                    ok = wait_bounded(&bar_rel[((n - NSLOT + 1) >> 1) % NREL],
                                      (uint32_t)(((n - NSLOT + 1) >> 1) / NREL) & 1u, abort_flag, p.status);
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
                const int j = key_tile(n >> 1);
                if (!p.ktl.sharded || j < p.ktl.g0) {
                    if (lane == 0) {  // a TMA tile: lane 0 alone
                        int kmap, khead, krow;
                        tile_src(p.ktl, p.W, j, r, h, p.Hl, kmap, khead, krow);
                        mbar_arrive_expect_tx(&bar_full[slot], SLOT);
                        const CUtensorMap *m = (n & 1) ? &p.tv[kmap] : &p.tk[kmap];
                        for (int db = 0; db < C::DB; db++)
                            tma_load_4d(&bar_full[slot], m, sbase + C::R_OFF + slot * C::TILE + db * 16384, db * 64,
                                        khead, krow, b);
                    }
                } else {
                    // a V slot this CTA has not filled yet gets its empty rows zeroed
                    fill_tail<D>(sbase + C::R_OFF + slot * C::TILE, p.ktl, p.W, j - p.ktl.g0,
                                 (n & 1) ? p.vptr : p.kptr, p.ks, b, r * p.Hl + h, lane, (n & 1) && use == 0);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar_full[slot]);
                }
            }
            if (lane == 0) {
                wait_drain(&bar_q, 0);
                for (int slot = 0; slot < NSLOT && slot < n; slot++) {
                    const int last = slot + ((n - 1 - slot) / NSLOT) * NSLOT;
                    wait_drain(&bar_full[slot], (uint32_t)(last / NSLOT) & 1u);
                }
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0 && nkv > 0) {
            constexpr int M = 128;
            constexpr uint32_t idesc_qk = make_idesc(M, 128, false);
            constexpr uint32_t idesc_pv = make_idesc(M, D, true);
            int issued = 0;
            // Descriptors are built once; a K step or a ring slot only moves the
            // 14-bit start-address field (shared-memory offsets are < 2^18, so the
            // field never carries into the next one).
            const uint64_t dq0 = make_sdesc(sbase + C::Q_OFF, 16, 1024);
            const uint64_t dq1 = make_sdesc(sbase + C::Q_OFF + C::TILE, 16, 1024);
            const uint64_t dk0 = make_sdesc(sbase + C::R_OFF, 16, 1024);  // K tile: K-major
            // V tile: MN-major (d contiguous), 8-key groups 1024 bytes apart, the
            // tile's two 64-column blocks 16 KB apart
            const uint64_t dv0 = make_sdesc(sbase + C::R_OFF, 16384, 1024);
            constexpr uint32_t kSlotStep = SLOT >> 4;
            // K-major column blocks: 16 KB apart
            constexpr int kBlk = 1024;
            auto qk = [&](int i, int slot) {
                const uint64_t a = i ? dq1 : dq0;
                const uint64_t bk = dk0 + (uint64_t)(slot * kSlotStep);
                const uint32_t d = tbase + (uint32_t)(i * 128);
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++) {
                    const uint64_t oa = (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2);  // Q: (kk/4)*16 KB + (kk%4)*32 B
                    const uint64_t ob = (uint64_t)((kk >> 2) * kBlk + (kk & 3) * 2);
                    mma_ss(d, a + oa, bk + ob, idesc_qk, kk > 0 ? 1u : 0u);
                }
                issued = 1;
            };
            auto pv = [&](int i, int slot, bool accumulate) {
                const uint64_t bv = dv0 + (uint64_t)(slot * kSlotStep);
                const uint32_t d = tbase + 256u + (uint32_t)(i * 128);
                const uint32_t pa = tbase + (uint32_t)(i * 128);
#pragma unroll
                for (int kk = 0; kk < 8; kk++) {  // 16 keys (2048 bytes of V) per step, all D columns at once
                    mma_ts(d, pa + (uint32_t)(kk * 8), bv + (uint64_t)(kk * 128), idesc_pv, (accumulate || kk > 0) ? 1u : 0u);
                }
                issued = 1;
            };
            auto signal = [&](uint64_t *bar) { mma_commit(bar); };
            // K of key tile j sits in slot (2j) % NSLOT, V in slot (2j+1) % NSLOT
            auto kslot = [](int j) { return (2 * j) % NSLOT; };
            // a slot is free once the MMAs that read it have completed
            auto vslot = [](int j) { return (2 * j + 1) % NSLOT; };
            auto kpar = [](int j) { return (uint32_t)((2 * j) / NSLOT) & 1u; };
            auto vpar = [](int j) { return (uint32_t)((2 * j + 1) / NSLOT) & 1u; };
            // a ring slot is ready when its barrier saw every byte
            auto slot_ready = [&](int slot, uint32_t par) {
                return wait_bounded(&bar_full[slot], par, abort_flag, p.status);
            };
            auto p_ready = [&](int i, uint32_t par) { return wait_bounded(&bar_pf[i], par, abort_flag, p.status); };
            bool ok = wait_bounded(&bar_q, 0, abort_flag, p.status) && slot_ready(kslot(0), kpar(0));
            if (ok) {
                tc_fence_after();
                qk(0, kslot(0));
                signal(&bar_sf[0]);
                qk(1, kslot(0));
                signal(&bar_sf[1]);
            }
            for (int jj = 0; ok && jj < nkv; jj++) {
                const bool more = jj + 1 < nkv;
                if (!slot_ready(vslot(jj), vpar(jj))) break;
                if (!p_ready(0, (uint32_t)jj & 1u)) break;
                tc_fence_after();
                pv(0, vslot(jj), jj > 0);
                if (more) {
                    if (!slot_ready(kslot(jj + 1), kpar(jj + 1))) break;
                    tc_fence_after();
                    qk(0, kslot(jj + 1));
                    signal(&bar_sf[0]);
                } else {
                    signal(&bar_of[0]);
                }
                if (!p_ready(1, (uint32_t)jj & 1u)) break;
                tc_fence_after();
                pv(1, vslot(jj), jj > 0);
                if (more) {
                    qk(1, kslot(jj + 1));
                    signal(&bar_sf[1]);
                } else {
                    signal(&bar_of[1]);
                }
            }
            if (*abort_flag && issued) {
                mma_commit(&bar_drain);
                wait_drain(&bar_drain, 0);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- softmax (warps 0-7)
        const int i = warp >> 2;       // query tile of the pair
        const int quarter = warp & 3;  // TMEM lane quarter
        const int row = quarter * 32 + lane;
        // global query token of this thread's row (>= Tq: the slot holds none)
        int q_row = qp * 256 + i * 128 + row;
        if (TILED) {
            q_row = tile_token(p.qtl, p.W, 2 * qp + i, row);
            if (q_row < 0) q_row = p.Tq;
        }
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS_me = tbase + lane_off + (uint32_t)(i * 128);
        const uint32_t tO_me = tbase + lane_off + 256u + (uint32_t)(i * 128);
        const float c = p.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        // Visibility bits of the tile to come are fetched while the tensor core
        // still works on it, never between S arriving and P leaving.
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        // sharded K/V without a mask: key tiles below kfull are whole tiles of real keys
        const int kfull = (TILED && p.ktl.sharded && p.mask_kind == SP_MASK_NONE) ? p.ktl.full0[p.W] : 0;
        auto tiled_words = [&](int j) {
            if (j < kfull) {
                w[0] = w[1] = w[2] = w[3] = 0xffffffffu;
            } else {
                const uint4 v = key_words_call(p, b, q_row, j, lane);
                w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
            }
        };
        // A key mask's bytes are loaded one tile before the tile whose bits
        // they give, so that the shuffles that gather them never wait on the load.
        const bool key_mask = !TILED && p.mask_kind == SP_MASK_KEY;
        uint32_t raw_next = 0u;
        if (nkv > 0) {
            if (TILED) tiled_words(key_tile(0));
            else mask_words(p, b, q_row, key_tile(0) * 128, lane, w);
            if (key_mask && nkv > 1) raw_next = mask_raw4(p.mask, key_tile(1) * 128 + 4 * lane, p.Tk, p.mask_vec4);
        }
        for (int jj = 0; jj < nkv; jj++) {
            const bool s_ok = wait_bounded(&bar_sf[i], (uint32_t)jj & 1u, abort_flag, p.status);
            if (!__all_sync(0xffffffffu, s_ok)) {  // leave together: the loop body is warp-collective
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[128];
            float mt;  // the row's maximum, reduced by the TMEM load itself
            tmem_ld_max_x128(tS_me, sr, mt);
            // the sharded instance relays release event jj as soon as S1(jj) is in
            if (TILED && i == 1 && quarter == 0 && lane == 0) mbar_arrive(&bar_rel[jj % NREL]);
            float *s = reinterpret_cast<float *>(sr);
            if ((w[0] & w[1] & w[2] & w[3]) != 0xffffffffu) {
                // some keys of the tile are hidden: mask them, then the maximum
                // is over the visible ones
#pragma unroll
                for (int e = 0; e < 128; e++)
                    if (!((w[e >> 5] >> (e & 31)) & 1u)) s[e] = -INFINITY;
                float m0 = fmaxf(s[0], s[1]), m1 = fmaxf(s[2], s[3]), m2 = fmaxf(s[4], s[5]), m3 = fmaxf(s[6], s[7]);
#pragma unroll
                for (int e = 8; e < 128; e += 8) {
                    m0 = fmax3(m0, s[e], s[e + 1]);
                    m1 = fmax3(m1, s[e + 2], s[e + 3]);
                    m2 = fmax3(m2, s[e + 4], s[e + 5]);
                    m3 = fmax3(m3, s[e + 6], s[e + 7]);
                }
                mt = fmax3(m0, m1, fmaxf(m2, m3));
            }
            float alpha = 1.f;
            if (mt > m) {
                if (m == -INFINITY) {
                    m = mt;  // no probability mass so far: O is zero
                } else if ((mt - m) * c > kRescaleThreshold) {
                    alpha = ex2((m - mt) * c);
                    m = mt;
                }
            }
            l *= alpha;
            const float mc = (m == -INFINITY) ? 0.f : m * c;
            uint32_t pk[64];
            // s * c - m * c and the four row-sum partials on packed pairs, two
            // lanes per instruction (each lane rounds as the scalar fmaf / fadd)
            const uint64_t c2 = f2_pack(c, c), nmc2 = f2_pack(-mc, -mc);
            uint64_t l01 = 0ull, l23 = 0ull;  // packed partial sums, lanes (0,1) and (2,3)
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                float x0, x1, x2, x3;
                f2_unpack(f2_fma(f2_pack_u(sr[2 * e], sr[2 * e + 1]), c2, nmc2), x0, x1);
                f2_unpack(f2_fma(f2_pack_u(sr[2 * e + 2], sr[2 * e + 3]), c2, nmc2), x2, x3);
                const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
                l01 = f2_add(l01, f2_pack(p0, p1));
                l23 = f2_add(l23, f2_pack(p2, p3));
                pk[e] = pack_bf16x2(p0, p1);
                pk[e + 1] = pack_bf16x2(p2, p3);
            }
            float l0, l1, l2, l3;
            f2_unpack(l01, l0, l1);
            f2_unpack(l23, l2, l3);
            l += (l0 + l1) + (l2 + l3);
            tmem_st_x64(tS_me, pk);  // P over the first 64 columns of S_i
            // O_i already holds PV_i(jj-1) (see the issue order above); rescale
            // it when the running max moved.  Warp-uniform: tcgen05.ld/st are
            // warp-collective, rows that did not move scale by 1.
            if (__any_sync(0xffffffffu, alpha != 1.f) && jj > 0) {
#pragma unroll
                for (int cc = 0; cc < D / 32; cc++) {
                    uint32_t o[32];
                    tmem_ld_x32(tO_me + cc * 32, o);
#pragma unroll
                    for (int e = 0; e < 32; e++) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st_x32(tO_me + cc * 32, o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar_pf[i]);
            if (jj + 1 < nkv) {
                if (TILED) {
                    tiled_words(key_tile(jj + 1));
                } else if (key_mask) {
                    nibbles_to_words(nibble_of(raw_next), lane, w);
                    if (jj + 2 < nkv) raw_next = mask_raw4(p.mask, key_tile(jj + 2) * 128 + 4 * lane, p.Tk, p.mask_vec4);
                } else {
                    mask_words(p, b, q_row, key_tile(jj + 1) * 128, lane, w);
                }
            }
            // S1(jj) was complete, so QK1(jj) and every MMA before it
            // (PV1(jj-1)) have completed: release event jj frees V(jj-1), K(jj)
            if (!TILED && i == 1 && quarter == 0 && lane == 0) mbar_arrive(&bar_rel[jj % NREL]);
        }
        // the epilogue has a 128-thread barrier: the tile's four warps decide together
        const bool epi = named_bar_and(1 + i, 128, ok && !*abort_flag);
        if (epi && qp < p.n_qpairs) {
            bool have = true;
            if (nkv > 0) {
                have = wait_bounded(&bar_of[i], 0, abort_flag, p.status);
                // the four warps decide together: the store below has a
                // 128-thread barrier that no warp may reach alone
                have = named_bar_and(1 + i, 128, have);
                tc_fence_after();
            }
            if (have) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
                int omap = r, ohead = h, orow = qp * 256 + i * 128;
                const bool whole = !TILED || tile_src(p.qtl, p.W, 2 * qp + i, r, h, p.Hl, omap, ohead, orow);
                if ((!SPLIT || piece < 0) && whole) {
                    uint8_t *tile = sgen + C::Q_OFF + i * C::TILE;
#pragma unroll
                    for (int db = 0; db < C::DB; db++) {
#pragma unroll
                        for (int half = 0; half < 2; half++) {
                            uint32_t o[32];
                            if (nkv > 0) {
                                tmem_ld_x32(tO_me + db * 64 + half * 32, o);
                            } else {
#pragma unroll
                                for (int e = 0; e < 32; e++) o[e] = 0u;
                            }
                            uint32_t pk[16];
#pragma unroll
                            for (int e = 0; e < 16; e++)
                                pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
#pragma unroll
                            for (int u = 0; u < 4; u++) {
                                const int chunk = half * 4 + u;
                                uint4 *dst = reinterpret_cast<uint4 *>(tile + db * 16384 + row * 128 +
                                                                       ((chunk ^ (row & 7)) << 4));
                                *dst = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(1 + i, 128);
                    if (quarter == 0 && lane == 0) {
                        for (int db = 0; db < C::DB; db++)
                            tma_store_4d(&p.to[omap], sbase + C::Q_OFF + i * C::TILE + db * 16384, db * 64, ohead,
                                         orow, b);
                        bulk_commit();
                        bulk_wait_read0();
                    }
                } else if (TILED && (!SPLIT || piece < 0)) {
                    // tail query tile: every thread stores its own row, if it holds a token
                    int s = 0, srow = 0;
                    const bool mine =
                        q_row < p.Tq && tiling_tail(p.qtl, p.W, (2 * qp + i - p.qtl.g0) * 128 + row, s, srow);
                    uint8_t *orow_ptr = mine ? p.optr[s] + ((int64_t)b * p.os[0] + (int64_t)srow * p.os[1] +
                                                            (int64_t)(r * p.Hl + h) * p.os[2]) * 2
                                             : nullptr;
#pragma unroll
                    for (int cc = 0; cc < D / 32; cc++) {
                        uint32_t o[32];
                        if (nkv > 0) {
                            tmem_ld_x32(tO_me + cc * 32, o);  // warp-collective: every lane loads
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; e++) o[e] = 0u;
                        }
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; e++)
                            pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                        if (mine) {
                            uint4 *dst = reinterpret_cast<uint4 *>(orow_ptr + cc * 64);
#pragma unroll
                            for (int u = 0; u < 4; u++)
                                dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                        }
                    }
                } else {
                    const int64_t prow = ((witem - p.n_full) * p.n_split + piece) * 256 + i * 128 + row;
                    float4 *dst = reinterpret_cast<float4 *>(p.part_o + prow * D);
#pragma unroll
                    for (int cc = 0; cc < D / 32; cc++) {
                        uint32_t o[32];
                        if (nkv > 0) {
                            tmem_ld_x32(tO_me + cc * 32, o);
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; e++) o[e] = 0u;
                        }
#pragma unroll
                        for (int e = 0; e < 8; e++)
                            dst[cc * 8 + e] =
                                make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                            __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
                    }
                    p.part_lse[prow] = l > 0.f ? m * c + log2f(l) : -INFINITY;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tbase, 512);
}

// Merge of split-key partials: one warp per (rank, batch, head, query) row.
struct MergeParams {
    void *o[SP_MAX_RANKS];
    int64_t os[3];
    int W, B, Tq, Hl, D, n_qpairs, n_split, n_full, n_pieced;
    Tiling qtl;  // sharded: o[s] are token shards (see TcParams)
    const float *part_o, *part_lse;
};

// Launched as a programmatic dependent of the attention kernel: its CTAs may
// be scheduled while the attention grid drains, and wait here until that grid
// has completed and its partials are visible.
template <int NJ>
__global__ void __launch_bounds__(256) attn_merge_kernel(MergeParams a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // one warp per output row of a pieced work item
    const int lane = threadIdx.x & 31;
    const int64_t rowid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (rowid >= (int64_t)a.n_pieced * 256) return;
    const int64_t pi = rowid >> 8;
    const int row = (int)(rowid & 255);
    int64_t t = a.n_full + pi;
    const int qp = (int)(t % a.n_qpairs);
    t /= a.n_qpairs;
    const int h = (int)(t % a.Hl);
    t /= a.Hl;
    const int b = (int)(t % a.B);
    const int r = (int)(t / a.B);
    int omap = r, ohead = h, orow = qp * 256 + row;
    if (!a.qtl.sharded) {
        if (orow >= a.Tq) return;
    } else {
        const int j = qp * 2 + (row >> 7), e = row & 127;
        int s, srow;
        int nvalid;
        if (tiling_box(a.qtl, a.W, j, s, srow, nvalid)) {
            if (e >= nvalid) return;  // past the end of a partial tile: no query
            srow += e;
        } else if (!tiling_tail(a.qtl, a.W, (j - a.qtl.g0) * 128 + e, s, srow)) {
            return;  // the slot holds no query
        }
        omap = s;
        ohead = r * a.Hl + h;
        orow = srow;
    }
    const int64_t item = pi;  // partials are indexed by pieced item
    float L = -INFINITY;
    for (int s = 0; s < a.n_split; s++) L = fmaxf(L, a.part_lse[(item * a.n_split + s) * 256 + row]);
    float acc[NJ];
#pragma unroll
    for (int j = 0; j < NJ; j++) acc[j] = 0.f;
    float wsum = 0.f;
    if (L != -INFINITY) {
        for (int s = 0; s < a.n_split; s++) {
            const int64_t prow = (item * a.n_split + s) * 256 + row;
            const float w = exp2f(a.part_lse[prow] - L);
            wsum += w;
#pragma unroll
            for (int j = 0; j < NJ; j++) acc[j] = fmaf(w, a.part_o[prow * a.D + lane + 32 * j], acc[j]);
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16 *O = (__nv_bfloat16 *)a.o[omap] + b * a.os[0] + (int64_t)orow * a.os[1] + ohead * a.os[2];
#pragma unroll
    for (int j = 0; j < NJ; j++) O[lane + 32 * j] = __float2bfloat16_rn(acc[j] * inv);
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static int get_encode() {
    if (g_encode) return SP_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return set_error(SP_ERR_CUDA, "cuTensorMapEncodeTiled unavailable: %s", cudaGetErrorString(e));
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    return SP_OK;
}

// 4-D map over (d, head, token, batch) with a 64 x 1 x 128 x 1 box, 128-byte swizzle.
static int encode_map(CUtensorMap *m, const void *base, int D, int Hl, int T, int B, const int64_t st[3]) {
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hl, (cuuint64_t)T, (cuuint64_t)B};
    // strides of a size-1 dim do not matter; give them a legal value
    int64_t hs = Hl > 1 ? st[2] : D, ts = T > 1 ? st[1] : (int64_t)Hl * hs, bs = B > 1 ? st[0] : (int64_t)T * ts;
    cuuint64_t strides[3] = {(cuuint64_t)hs * 2, (cuuint64_t)ts * 2, (cuuint64_t)bs * 2};
    cuuint32_t box[4] = {64, 1, 128, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult rc = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (rc != CUDA_SUCCESS) return set_error(SP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)rc);
    return SP_OK;
}

// Real rows of shard s of an operand of T tokens in shards of Tl (the
// operand's own T rows when it is not sharded, Tl == 0).
static int map_rows(int Tl, int T, int s) {
    if (Tl <= 0) return T;
    const int64_t n = (int64_t)T - (int64_t)s * Tl;
    return (int)(n < 0 ? 0 : (n > Tl ? Tl : n));
}

static void make_tiling(Tiling &t, int Tl, int T, int W) {
    memset(&t, 0, sizeof(t));
    if (Tl <= 0) return;
    t.sharded = 1;
    t.Tl = Tl;
    for (int s = 0; s < W; s++) {
        const int n = map_rows(Tl, T, s), rem = n % 128;
        const bool partial = rem >= kPartialMin;
        t.rows[s] = n;
        if (partial) t.part[t.npart++] = s;
        t.full0[s + 1] = t.full0[s] + n / 128;
        t.tail0[s + 1] = t.tail0[s] + (partial ? 0 : rem);
    }
    t.g0 = t.full0[W] + t.npart;
}

// Work decomposition.  A work item is one (rank, batch, head, query pair); a
// CTA holds one SM (225 KB of shared memory), so items run in waves of
// num_SMs.  Two cases cut items into key pieces (merged by LSE afterwards):
//  - fewer items than SMs (short query sequences): every item, into enough
//    pieces to fill the SMs, at least 4 key tiles each;
//  - a last, partial wave: only its items, into the piece count that finishes
//    soonest, counting each unit's fixed cost (Q load, epilogue, merge) as
//    four key tiles; kept only when the whole launch gets 3 % shorter.
struct SplitPlan {
    int n_qpairs, n_kv;
    int n_full, n_pieced;  // items run whole / items cut into n_split pieces
    int n_split, kv_per_split;
    size_t extra_bytes;
};

static SplitPlan plan_split(int W, int B, int Tq, int Tk, int Hl, int D, int num_sms) {
    SplitPlan s;
    s.n_qpairs = (Tq + 255) / 256;
    s.n_kv = (Tk + 127) / 128;
    const int64_t items = (int64_t)W * B * Hl * s.n_qpairs;
    s.n_full = (int)items;
    s.n_pieced = 0;
    int ns = 1;
    if (items > 0 && items < num_sms && s.n_kv >= 8) {
        ns = (int)(num_sms / items);
        const int cap = s.n_kv / 4;  // at least 4 key tiles per split
        if (ns > cap) ns = cap;
        if (ns < 1) ns = 1;
        if (ns > 1) {
            s.n_full = 0;
            s.n_pieced = (int)items;
        }
    } else if (items > num_sms && s.n_kv >= 8) {
        const int64_t tail = items % num_sms;
        const double kFixed = 4.0;  // per-unit cost in key tiles (Q load, epilogue, merge)
        const double whole = s.n_kv + kFixed;
        double best = whole;
        for (int c = 2; c <= 8 && tail > 0; c++) {
            const int per = (s.n_kv + c - 1) / c;
            if (per < 4) break;
            const double cost = (double)((tail * c + num_sms - 1) / num_sms) * (per + kFixed);
            if (cost < best) {
                best = cost;
                ns = c;
            }
        }
        // worth it only if the whole launch gets at least 3 % shorter
        const double full_waves = (double)(items / num_sms);
        if (ns > 1 && full_waves * whole + best < 0.97 * (full_waves + 1.0) * whole) {
            s.n_full = (int)(items - tail);
            s.n_pieced = (int)tail;
        } else {
            ns = 1;
        }
    }
    s.kv_per_split = s.n_kv > 0 ? (s.n_kv + ns - 1) / ns : 1;
    s.n_split = s.n_kv > 0 ? (s.n_kv + s.kv_per_split - 1) / s.kv_per_split : 1;
    if (s.n_split <= 1) {
        s.n_split = 1;
        s.n_full = (int)items;
        s.n_pieced = 0;
    }
    s.extra_bytes = s.n_pieced > 0 ? (size_t)s.n_pieced * s.n_split * 256 * (size_t)(D + 1) * sizeof(float) : 0;
    return s;
}

}  // namespace tc

size_t attn_tc_extra_bytes(int W, int B, int Tq, int Tk, int Hl, int D) {
    DeviceInfo di;
    if (device_info(&di) != SP_OK) return 0;
    return tc::plan_split(W, B, Tq, Tk, Hl, D, di.num_sms).extra_bytes;
}

bool attn_tc_supported(const AttnArgs &a) {
    if (a.dtype != SP_BF16 || (a.D != 64 && a.D != 128) || a.Tq <= 0 || a.Tk <= 0) return false;
    for (int i = 0; i < 3; i++)
        if (((a.qs[i] | a.ks[i] | a.os[i]) * 2) % 16 != 0) return false;
    for (int r = 0; r < a.W; r++)
        if (((uintptr_t)a.q[r] | (uintptr_t)a.k[r] | (uintptr_t)a.v[r] | (uintptr_t)a.o[r]) & 15) return false;
    return true;
}

template <int D, bool SPLIT, bool TILED>
static int launch_tc_t(const tc::TcParams &prm, unsigned grid, cudaStream_t st) {
    // the shared-memory opt-in is a per-device attribute of each instance: set
    // once per device (a bit per device; a racing second set is harmless)
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    SP_CUDA_CHECK(cudaGetDevice(&dev));
    auto kern = tc::attn_tc_kernel<D, SPLIT, TILED>;
    const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        SP_CUDA_CHECK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::Cfg<D>::SMEM_ALLOC));
        configured.fetch_or(bit, std::memory_order_release);
    }
    kern<<<grid, tc::kThreads, tc::Cfg<D>::SMEM_ALLOC, st>>>(prm);
    return check_launch("sp_attention(tcgen05)");
}

int launch_attn_tc(const AttnArgs &a, cudaStream_t st) {
    int rc = tc::get_encode();
    if (rc) return rc;
    DeviceInfo di;
    rc = device_info(&di);
    if (rc) return rc;
    if (di.cc_major != 10) return set_error(SP_ERR_UNSUPPORTED, "tcgen05 path needs a Blackwell (sm_10x) device");
    static thread_local tc::TcParams prm;  // 4+ KB: keep it off the stack
    memset(&prm, 0, sizeof(prm));
    // per-rank tensors: [B, T, Hl, D]; token shards: [B, n_s, W*Hl, D], shard s
    // holding its n_s real rows (maps end there: a shard may be a view that
    // stops at the caller's last token)
    tc::make_tiling(prm.qtl, a.q_shard_rows, a.Tq, a.W);
    tc::make_tiling(prm.ktl, a.kv_shard_rows, a.Tk, a.W);
    const int qh = a.q_shard_rows > 0 ? a.W * a.Hl : a.Hl, kh = a.kv_shard_rows > 0 ? a.W * a.Hl : a.Hl;
    for (int r = 0; r < a.W; r++) {
        const int qt = tc::map_rows(a.q_shard_rows, a.Tq, r), kt = tc::map_rows(a.kv_shard_rows, a.Tk, r);
        // a shard with no rows is never read: its map repeats shard 0's
        const int rq = qt > 0 ? r : 0, rk = kt > 0 ? r : 0;
        const int nq = qt > 0 ? qt : tc::map_rows(a.q_shard_rows, a.Tq, 0);
        const int nk = kt > 0 ? kt : tc::map_rows(a.kv_shard_rows, a.Tk, 0);
        if ((rc = tc::encode_map(&prm.tq[r], a.q[rq], a.D, qh, nq, a.B, a.qs))) return rc;
        if ((rc = tc::encode_map(&prm.tk[r], a.k[rk], a.D, kh, nk, a.B, a.ks))) return rc;
        if ((rc = tc::encode_map(&prm.tv[r], a.v[rk], a.D, kh, nk, a.B, a.ks))) return rc;
        if ((rc = tc::encode_map(&prm.to[r], a.o[rq], a.D, qh, nq, a.B, a.os))) return rc;
        prm.qptr[r] = (const uint8_t *)a.q[r];
        prm.kptr[r] = (const uint8_t *)a.k[r];
        prm.vptr[r] = (const uint8_t *)a.v[r];
        prm.optr[r] = (uint8_t *)a.o[r];
    }
    for (int i = 0; i < 3; i++) {
        prm.qs[i] = a.qs[i];
        prm.ks[i] = a.ks[i];
        prm.os[i] = a.os[i];
    }
    const bool tiled = a.q_shard_rows > 0 || a.kv_shard_rows > 0;
    // Tiles of each operand.  A sharded one can have more than ceil(T / 128):
    // every shard whose leftover block holds >= kPartialMin rows adds a partial
    // tile of its own (up to W more in all), so the work decomposition counts
    // the tiling's tiles, not the tokens.
    auto n_tiles = [&](const tc::Tiling &t, int T) {
        return t.sharded ? t.g0 + (t.tail0[a.W] + 127) / 128 : (T + 127) / 128;
    };
    const int q_tiles = n_tiles(prm.qtl, a.Tq), kv_tiles = n_tiles(prm.ktl, a.Tk);
    tc::SplitPlan sp = tc::plan_split(a.W, a.B, q_tiles * 128, kv_tiles * 128, a.Hl, a.D, di.num_sms);
    if (sp.n_split > 1 && (a.extra == nullptr || a.extra_bytes < sp.extra_bytes)) {
        sp.n_split = 1;
        sp.kv_per_split = sp.n_kv > 0 ? sp.n_kv : 1;
        sp.n_full = a.W * a.B * a.Hl * sp.n_qpairs;
        sp.n_pieced = 0;
        sp.extra_bytes = 0;
    }
    prm.W = a.W;
    prm.B = a.B;
    prm.Tq = a.Tq;
    prm.Tk = a.Tk;
    prm.Hl = a.Hl;
    prm.n_qpairs = sp.n_qpairs;
    prm.n_kv = sp.n_kv;
    prm.n_split = sp.n_split;
    prm.kv_per_split = sp.kv_per_split;
    prm.n_full = sp.n_full;
    prm.scale_log2 = a.scale * 1.4426950408889634f;
    prm.mask_kind = a.mask_kind;
    prm.mask = a.mask;
    // 4-byte mask reads need 4-aligned key runs: every whole key tile of a
    // sharded K/V starts at a multiple of the shard length
    prm.mask_vec4 =
        (a.mask && ((uintptr_t)a.mask & 3) == 0 && (a.Tk & 3) == 0 && (a.kv_shard_rows & 3) == 0) ? 1 : 0;
    prm.status = &a.ws->status;
    prm.kv_stall = &a.ws->kv_stall;
    const int64_t grid = sp.n_split > 1 ? (int64_t)sp.n_full + (int64_t)sp.n_pieced * sp.n_split
                                        : (int64_t)a.W * a.B * a.Hl * sp.n_qpairs;
    if (grid == 0) return SP_OK;
    if (grid > 0x7fffffffll) return set_error(SP_ERR_INVALID_ARG, "sp_attention: grid too large");
    if (sp.n_split > 1) {
        prm.part_o = reinterpret_cast<float *>(a.extra);
        prm.part_lse = prm.part_o + (size_t)sp.n_pieced * sp.n_split * 256 * a.D;
        rc = (a.D == 64) ? (tiled ? launch_tc_t<64, true, true>(prm, (unsigned)grid, st)
                                  : launch_tc_t<64, true, false>(prm, (unsigned)grid, st))
                         : (tiled ? launch_tc_t<128, true, true>(prm, (unsigned)grid, st)
                                  : launch_tc_t<128, true, false>(prm, (unsigned)grid, st));
        if (rc) return rc;
        tc::MergeParams mp;
        memset(&mp, 0, sizeof(mp));
        for (int r = 0; r < a.W; r++) mp.o[r] = a.o[r];
        for (int i = 0; i < 3; i++) mp.os[i] = a.os[i];
        mp.W = a.W;
        mp.B = a.B;
        mp.Tq = a.Tq;
        mp.Hl = a.Hl;
        mp.D = a.D;
        mp.n_qpairs = sp.n_qpairs;
        mp.n_split = sp.n_split;
        mp.n_full = sp.n_full;
        mp.n_pieced = sp.n_pieced;
        mp.qtl = prm.qtl;
        mp.part_o = prm.part_o;
        mp.part_lse = prm.part_lse;
        const int64_t rows = (int64_t)sp.n_pieced * 256;
        const unsigned blocks = (unsigned)((rows * 32 + 255) / 256);
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = dim3(blocks, 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = (a.D == 64) ? cudaLaunchKernelEx(&cfg, tc::attn_merge_kernel<2>, mp)
                                    : cudaLaunchKernelEx(&cfg, tc::attn_merge_kernel<4>, mp);
        if (e != cudaSuccess)
            return set_error(SP_ERR_CUDA, "sp_attention(merge) launch failed: %s", cudaGetErrorString(e));
        return check_launch("sp_attention(merge)");
    }
    if (a.D == 64)
        return tiled ? launch_tc_t<64, false, true>(prm, (unsigned)grid, st)
                     : launch_tc_t<64, false, false>(prm, (unsigned)grid, st);
    return tiled ? launch_tc_t<128, false, true>(prm, (unsigned)grid, st)
                 : launch_tc_t<128, false, false>(prm, (unsigned)grid, st);
}

}  // namespace sp
