// dense_block_tc.cu - the dense-masked attention block of the block page's
// module shape (Kimi-K2.6 l2_p4, reference model: P = 16 pair features,
// H = 4 heads of 24 dims, D = 96, up to 24 nodes): the four D x D projections
// and the relation MLP's first layer on the 5th-generation tensor cores
// (tcgen05, kind::f16, fp32 accumulators in TMEM), the attention's Q K^T and
// A V on warp-level f16 MMAs, the rest in fp32 on the CUDA cores.
//
// Tensor-core precision: fp32 results from fp16 products. Each operand row (a
// normalised node row, a Q / K / V / context row, a pair's features, a weight
// matrix, the attention weights) is scaled by a power of two 2^s that brings
// its largest magnitude into [2^12, 2^13), then split x 2^s = hi + lo,
// hi = fp16(x 2^s) and lo = fp16(x 2^s - hi) (round to nearest even).
// A B ~ hi_A hi_B + hi_A lo_B + lo_A hi_B: the dropped lo_A lo_B and lo's own
// rounding are ~2^-22 of the row's largest term, the products accumulate in
// fp32, and the scales are undone exactly afterwards. Three fp16 MMAs cost
// what 1.5 tf32 MMAs do, for the accuracy of the 3xTF32 split.
//
// The projections' A operands live in TMEM (written by tcgen05.st from the
// registers of the threads owning the row), so those tensor cores read only
// the weights from shared memory. A tile is 4 graphs padded to 32 rows: graph
// g owns TMEM lanes 32g..32g+31, which warps g, g+4, g+8, g+12 may access.
// Every projection MMA is 128 x 96 x 16 (a tcgen05 MMA costs ~47 cycles at any
// N up to 96, so wide MMAs and few of them): Q, K, V and the out-projection
// are 18 MMAs each.
//
// 17 warps per CTA, one CTA per SM, persistent over tiles; per tile t:
//   control warp (lane 0): streams the pre-split weight chunks (K Q V O, 96
//       rows each) through a 2-slot shared-memory ring with bulk copies and
//       issues them: K and V once LayerNorm(t) is in TMEM, Q once tile t-1's
//       epilogue has read the out-projection from its columns, the
//       out-projection once the context is; it also bulk-copies the next
//       tile's node rows;
//   A (quad q = warps 4q..4q+3): the relation MLP over the tile's unmasked
//       pairs only (a masked pair's logit is -inf whatever its bias, so its
//       features are never read): per (graph, query row) a word of unmasked
//       keys and a prefix of their counts, built from the mask in shared
//       memory during the tile before; one thread per unmasked pair of
//       128-pair blocks q, q + 4, ...: the pair's 16 features (prefetched into
//       shared memory by cp.async) go, split and scaled, to its TMEM lane as
//       the A operand of W1 (128 x 16 x 16 MMAs the quad's first thread
//       issues, in TMEM columns idle until the next tile's LayerNorm); the
//       same thread reads the hidden values back and applies b1, SiLU, W2, b2
//       (packed f32x2 FMAs), giving the bias of all heads;
//   B (warp (g, h) = (w % 4, w / 4)): attention of head h in graph g on
//       warp-level MMAs (m16n8k16, f16 operands split in two, three products
//       per term): Q and K fragments loaded straight from TMEM (16x256b),
//       each row scaled from its own range; bias in log2 units (-inf for the
//       query's masked keys, from its word), softmax with ex2 over the quad
//       of lanes sharing a row; A V with V staged in shared memory; the
//       context stored from the fragments (16x128b) as the out-projection's A
//       operand (scaled per graph by the largest |V|, which bounds it); the
//       next tile's mask (copied in during B) becomes its unmasked-pair words;
//   C: LayerNorm of tile t+1 into the other A region of TMEM (warp (g, k):
//       columns [24k, 24k + 24) of graph g's rows, row statistics combined
//       through shared memory) with tile t+1's pair prefix, its first
//       relation-MLP prefetches and tile t's residual rows copied in; then
//       the epilogue per graph: the four head warps add their out-projection
//       columns to the staged residual block, and its 128 threads store the
//       block as consecutive float4s.
// Every mbarrier wait is bounded; a wait that gives up sets the call's error
// flag in the workspace (readable with gat_dense_masked_attention_status) and
// the outputs of the remaining tiles are written as NaN, never as garbage.
#include <cuda_fp16.h>

#include "common.cuh"

namespace gat {

namespace tc {

constexpr int P = 16, H = 4, DH = 24, D = H * DH;
constexpr int kComputeWarps = 16;
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kThreads = kComputeThreads + 32;  // + the control warp
constexpr int kGraphs = 4;                        // graphs per tile
constexpr int kMaxN = 24;                         // nodes per graph (shared memory bound)
constexpr int kChunks = 4;                        // weight chunks per tile: Q K V O
constexpr int kRing = 2;
constexpr uint32_t kChunkHalf = D * D * 2;        // one of hi / lo, fp16
constexpr uint32_t kChunkBytes = 2 * kChunkHalf;
constexpr uint32_t kW1Half = P * P * 2;           // W1 image, one of hi / lo
// staged node rows: stride 100 floats, so the 16-byte loads of 8 lanes
// (8 consecutive rows) fall in 8 distinct bank quads (one bulk copy per row)
constexpr int kNodeStride = D + 4;
// staged output rows: the same stride (8 consecutive rows' 16-byte stores in
// 8 distinct bank quads)
constexpr int kOutStride = D + 4;
// row stride of the relation-MLP bias: at least N + 1 and 12 mod 16, so that
// the attention's fragment reads (keys 2 apart in a quad of lanes, rows
// consecutive) fall in distinct banks
__host__ __device__ constexpr int bias_stride(int N) { return N + 1 + ((12 - (N + 1)) & 15); }
// residual / output float4s per thread of a graph's 128 (warps g, g + 4, ...)
constexpr int kOutVec = (kMaxN * D / 4 + 127) / 128;
// TMEM columns (32-bit): fp32 accumulators, or fp16 pairs for A operands
// A operands (x_n, then the context) at column 288 (even tiles) or 384 (odd)
// (hi: kAHalf columns of fp16 pairs for the D inputs, then lo)
__host__ __device__ constexpr uint32_t col_a(int t) { return (t & 1) ? 384u : 288u; }
constexpr uint32_t kAHalf = D / 2;
// relation-MLP slot of quad q in tile t: A hi (8) | A lo (8) | D (16) columns,
// in the next tile's A region (idle until its LayerNorm) or columns 480-511
__host__ __device__ constexpr uint32_t mlp_col(int t, int q) {
    return q < 3 ? col_a(t + 1) + 32u * q : 480u;
}
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 1000000000ull;       // a wait gives up after 1 s (never expected)
constexpr float kLog2e = 1.4426950408889634f;

// Workspace written by the prep kernel: header, then the weight images.
constexpr size_t kWsChunks = 256;
constexpr size_t kWsW1 = kWsChunks + (size_t)kChunks * kChunkBytes;
constexpr size_t kWsBytes = kWsW1 + 2 * kW1Half;
struct WsHeader {
    int32_t sw[5];  // scale exponents of Wq, Wk, Wv, Wout, W1
    int32_t err;    // set when a bounded wait gives up
};

// ---------------------------------------------------------------------------
// small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 2^s for |s| <= 126, exact
__device__ __forceinline__ float exp2i(int s) { return __int_as_float((127 + s) << 23); }

// scale exponent s with m 2^s in [2^12, 2^13) (0 for m = 0 or not finite)
__device__ __forceinline__ int scale_exp(float m) {
    if (!(m > 0.f) || !(m < INFINITY)) return 0;
    const int e = ilogbf(m);
    int s = 12 - e;
    return s < -120 ? -120 : (s > 120 ? 120 : s);
}

// (x0, x1) -> packed fp16 hi pair and lo pair (element x0 in the low half)
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// byte offset of element (r, k) of a K-major fp16 operand with K columns:
// 8-row x 16-byte core matrices, K-adjacent ones 128 bytes apart
__host__ __device__ __forceinline__ uint32_t kmaj16(int r, int k, int K) {
    return (uint32_t)((r >> 3) * (K >> 3) * 128 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}

// instruction descriptor: fp32 accumulate, fp16 A and B, both K-major
__host__ __device__ constexpr uint32_t idesc_f16(int n, int m) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D (tmem) (+)= A (tmem) B^T (smem)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                       int acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool flag_set(const int32_t *err) {
    return *reinterpret_cast<const volatile int32_t *>(err) != 0;
}

// Bounded wait for the phase of parity `parity`: false when it gives up,
// after kWaitNs (raising the error flag), or at once when an earlier wait of
// this call already gave up and `honor_err` is set (the pipeline is broken;
// the outputs become NaN, and the rest of the kernel runs through quickly).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int32_t *err,
                                          bool honor_err = true) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (done) return true;
        if ((it & 63) == 63) {
            if (honor_err && flag_set(err)) return false;
            const uint64_t t = now_ns();
            if (t0 == 0) {
                t0 = t;
            } else if (t - t0 > kWaitNs) {
                atomicExch(err, 1);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 8 / 16 consecutive TMEM columns of this warp's 32 lanes
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float *v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 TMEM lanes x 8 columns (16x256b shape): thread t gets lane base + t / 4
// at columns 2 (t % 4) and 2 (t % 4) + 1 (r[0], r[1]) and lane base + 8 + t / 4
// at the same columns (r[2], r[3]); no wait (the tied waits below)
__device__ __forceinline__ void tmem_ld16x8(uint32_t taddr, uint32_t *r) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}
// the wait for this thread's TMEM loads, with the loads' registers tied to it
// so that no use moves above it
__device__ __forceinline__ void tmem_wait_tied(uint32_t *a, uint32_t *b) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(b[0]), "+r"(b[1]),
                   "+r"(b[2]), "+r"(b[3])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_tied(uint32_t *a, uint32_t *b, uint32_t *c, uint32_t *d) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(b[0]), "+r"(b[1]),
                   "+r"(b[2]), "+r"(b[3]), "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3]),
                   "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
                 :
                 : "memory");
}

// 16 TMEM lanes x 4 columns (16x128b shape): thread t writes lane
// base + t / 4 at column t % 4 (a) and lane base + 8 + t / 4 there (b)
__device__ __forceinline__ void tmem_st16x4(uint32_t taddr, uint32_t a, uint32_t b) {
    asm volatile("tcgen05.st.sync.aligned.16x128b.x1.b32 [%0], {%1,%2};" ::"r"(taddr), "r"(a), "r"(b)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t *r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

// this thread's TMEM stores are complete and ordered before a later thread sync
__device__ __forceinline__ void tmem_st_done() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    fence_before();
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}


__device__ __forceinline__ uint64_t pk2(float2 v) { return *reinterpret_cast<uint64_t *>(&v); }
__device__ __forceinline__ float2 up2(uint64_t v) { return *reinterpret_cast<float2 *>(&v); }

// packed fp32 FMA on a pair: (a.x b.x + c.x, a.y b.y + c.y), each rounded once
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)), "l"(pk2(c)));
    return up2(r);
}

// d += A B for one warp: A 16 x 16 (row-major fragment), B 16 x 8
// (column-major fragment), f16 operands (element pairs packed low first),
// fp32 accumulators
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4],
                                        const uint32_t (&b)[2]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// ---------------------------------------------------------------------------
// prep: weights -> scaled fp16 hi / lo images in the shared-memory layout
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 256;

// Block m: matrix m of (Wq, Wk, Wv, Wout, W1), all rows.
__global__ void __launch_bounds__(kPrepThreads)
dense_prep_kernel(const float *__restrict__ Wq, const float *__restrict__ Wk,
                  const float *__restrict__ Wv, const float *__restrict__ Wout,
                  const float *__restrict__ W1, unsigned char *__restrict__ ws) {
    __shared__ float red[kPrepThreads / 32];
    const int m = blockIdx.x, tid = threadIdx.x;
    const float *W = m == 0 ? Wq : m == 1 ? Wk : m == 2 ? Wv : m == 3 ? Wout : W1;
    const int K = m < 4 ? D : P;  // square matrices
    float mx = 0.f;
    for (int i = tid; i < K * K; i += kPrepThreads) mx = fmaxf(mx, fabsf(__ldg(W + i)));
    mx = warp_max(mx);
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    mx = 0.f;
#pragma unroll
    for (int w = 0; w < kPrepThreads / 32; ++w) mx = fmaxf(mx, red[w]);
    const int s = scale_exp(mx);
    WsHeader *hd = reinterpret_cast<WsHeader *>(ws);
    if (tid == 0) {
        hd->sw[m] = s;
        if (m == 0) hd->err = 0;
    }
    const float sc = exp2i(s);
    unsigned char *dst = ws + (m < 4 ? kWsChunks + (size_t)m * kChunkBytes : kWsW1);
    const uint32_t half = m < 4 ? kChunkHalf : kW1Half;
    for (int i = tid; i < K * K / 2; i += kPrepThreads) {
        const int n = i / (K / 2), k = 2 * (i % (K / 2));
        const float *src = W + (int64_t)n * K + k;
        uint32_t hi, lo;
        split2(__ldg(src) * sc, __ldg(src + 1) * sc, hi, lo);
        const uint32_t off = kmaj16(n, k, K);
        *reinterpret_cast<uint32_t *>(dst + off) = hi;
        *reinterpret_cast<uint32_t *>(dst + half + off) = lo;
    }
}

// ---------------------------------------------------------------------------
// main kernel
// ---------------------------------------------------------------------------
struct Params {
    int32_t B, N;
    const float *nodes, *pair, *mask, *ln_w, *ln_b;
    float ln_eps;
    const float *W1, *b1, *W2, *b2;
    const unsigned char *ws;
    float *out;
};

// dynamic shared memory carve-up (bytes) for N nodes per graph
struct Smem {
    static constexpr uint32_t ring = 0;
    static constexpr uint32_t bias = ring + kRing * kChunkBytes;
    // relation-MLP bias (and scores) [graph][head][j][node, row stride bias_stride(N)];
    // between the attention and the next relation MLP it holds the LayerNorm
    // row statistics [sum | sum sq | max dev][4 column quarters][128 rows]
    static constexpr uint32_t lnred_bytes = 3 * 4 * 128 * 4;
    __host__ __device__ static uint32_t bias_bytes(int N) {
        const uint32_t b = kGraphs * H * N * bias_stride(N) * 4;
        return b > lnred_bytes ? b : lnred_bytes;
    }
    __host__ __device__ static uint32_t stage(int N) { return bias + bias_bytes(N); }
    // the attention's staging (per warp: the V rows), or outside it one
    // prefetch slot of 16
    // features per compute thread; above both (float offset mask_off), the
    // next tile's mask values, copied in during the attention. The epilogue's
    // output rows [graph][node][kOutStride] sit above the prefetch slots
    // (float offset out_off), over the attention's staging and the mask
    // values, both idle then.
    __host__ __device__ static uint32_t warp_stage(int N) { return N * DH; }
    __host__ __device__ static uint32_t mask_off(int N) {
        const uint32_t att = kComputeWarps * warp_stage(N), mlp = kComputeThreads * P;
        return att > mlp ? att : mlp;
    }
    static constexpr uint32_t out_off = kComputeThreads * P;
    __host__ __device__ static uint32_t stage_bytes(int N) {
        const uint32_t a = mask_off(N) + kGraphs * N * N, o = out_off + kGraphs * N * kOutStride;
        return (a > o ? a : o) * 4;
    }
    __host__ __device__ static uint32_t nodes(int N) { return stage(N) + stage_bytes(N); }
    __host__ __device__ static uint32_t nodes_bytes(int N) { return kGraphs * N * kNodeStride * 4; }
    // W1 image (fp16 hi | lo, the MMA's B operand), b1, W2 transposed [u][h], b2,
    // gamma, beta, max |gamma|, max |beta|
    __host__ __device__ static uint32_t params(int N) { return nodes(N) + nodes_bytes(N); }
    static constexpr uint32_t params_bytes = (P * P + P + P * H + H + 2 * D + 4) * 4;
    __host__ __device__ static uint32_t rscale(int N) { return params(N) + params_bytes; }
    // the tile's unmasked pairs: per (graph, query row) a word of unmasked
    // keys (bit j), and the exclusive prefix of their counts over the 128
    // rows (graph-major), [128] = the tile's total
    __host__ __device__ static uint32_t umask(int N) { return rscale(N) + 128 * 4; }
    __host__ __device__ static uint32_t rpre(int N) { return umask(N) + 128 * 4; }
    __host__ __device__ static uint32_t total(int N) { return rpre(N) + 132 * 4; }
};

struct Barriers {
    uint64_t wfull[kRing], wdone[kRing], dfull[4], nfull, xfull, edone, qk, vdone, cfull, ofull, drain;
};

// Control thread: weight ring and every MMA issue, driven by mbarriers.
// Per tile the weight chunks stream as K, Q, V, O (workspace images 1, 0, 2,
// 3; ring slots 0, 1, 0, 1): K and V (TMEM columns 96-287) go as soon as the
// tile's LayerNorm is in TMEM, since the previous tile's attention - their
// only other reader - is over by then; Q (columns 0-95) waits for the
// previous tile's epilogue to read the out-projection there, its weights
// loaded long before into the slot the previous O freed; O for the context.
// The scores wait for K and Q (one commit after Q), the context for V.
__host__ __device__ constexpr int chunk_of(int pos) { return pos == 0 ? 1 : pos == 1 ? 0 : pos == 2 ? 2 : 3; }

__device__ void control_loop(const Params &p, unsigned char *sm, Barriers &br, uint32_t tmem,
                             int n_my, const float *nodes_s, int32_t *err) {
    const int total = kChunks * n_my;
    uint32_t ph_wfull = 0, ph_wdone = 0;  // expected parity per ring slot, one bit each
    const unsigned char *src0 = p.ws + kWsChunks;
    const uint32_t ring0 = smem_u32(sm + Smem::ring);
    auto load = [&](int r) {
        const int s = r % kRing;
        const uint32_t bar = smem_u32(&br.wfull[s]);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"(kChunkBytes)
                     : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
            "[%3];" ::"r"(ring0 + (uint32_t)s * kChunkBytes),
            "l"(src0 + (size_t)chunk_of(r % kChunks) * kChunkBytes), "r"(kChunkBytes), "r"(bar)
            : "memory");
    };
    int loaded = 0, issued = 0, refill = 0;
    for (; loaded < total && loaded < kRing; ++loaded) load(loaded);
    constexpr uint32_t idesc = idesc_f16(D, 128);
    // a tile's node rows (contiguous graphs) into the staging buffer, one
    // bulk copy per row (rows kNodeStride floats apart)
    auto load_nodes = [&](int tl) {
        const int64_t b0 = (int64_t)tl * kGraphs;
        const int64_t ng = p.B - b0 < kGraphs ? p.B - b0 : kGraphs;
        const int rows = (int)(ng * p.N);
        const uint32_t bar = smem_u32(&br.nfull);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"((uint32_t)(rows * D * 4))
                     : "memory");
        const float *src = p.nodes + b0 * p.N * D;
        const uint32_t dst = smem_u32(nodes_s);
        for (int r = 0; r < rows; ++r)
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
                "[%3];" ::"r"(dst + (uint32_t)(r * kNodeStride * 4)),
                "l"(src + (int64_t)r * D), "r"((uint32_t)(D * 4)), "r"(bar)
                : "memory");
    };
    if (n_my > 0) load_nodes(blockIdx.x);
    bool bail = false;
    for (int t = 0; t < n_my && !bail; ++t) {
        // K, V(t) overwrite columns [96, 288) that tile t-1's attention read
        // (over: its context was signalled before O(t-1) was issued) and Q(t)
        // columns [0, 96) that its epilogue reads: LayerNorm(t) for all
        // three, tile t-1's epilogue for Q
        bool x_ok = false, e_ok = t == 0, c_ok = false;
        uint64_t idle_since = 0;
        uint32_t idle = 0;
        const uint32_t acol = col_a(t);
        while (issued < kChunks * (t + 1)) {
            bool progress = false;
            if (refill < issued && loaded < total) {
                const int s = refill % kRing;
                if (mbar_test(&br.wdone[s], (ph_wdone >> s) & 1u)) {
                    ph_wdone ^= 1u << s;
                    load(loaded++);
                    ++refill;
                    progress = true;
                }
            }
            {
            const int pos = issued % kChunks, c = chunk_of(pos), s = issued % kRing;
            if (!x_ok) x_ok = mbar_test(&br.xfull, (uint32_t)t & 1u);
            if (!e_ok) e_ok = mbar_test(&br.edone, (uint32_t)(t - 1) & 1u);
            if (c == kChunks - 1 && !c_ok) c_ok = mbar_test(&br.cfull, (uint32_t)t & 1u);
            const bool ready = c == kChunks - 1 ? c_ok : (c == 0 ? x_ok && e_ok : x_ok);
            if (ready && mbar_test(&br.wfull[s], (ph_wfull >> s) & 1u)) {
                ph_wfull ^= 1u << s;
                fence_after();
                const uint32_t bh = ring0 + (uint32_t)s * kChunkBytes, bl = bh + kChunkHalf;
                const uint32_t d = tmem + (uint32_t)(c < kChunks - 1 ? D * c : 0);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t ah = tmem + acol + 8u * ks, al = ah + kAHalf;
                    const uint64_t dh = smem_desc(bh + 256u * ks, 128, (D / 8) * 128);
                    const uint64_t dl = smem_desc(bl + 256u * ks, 128, (D / 8) * 128);
                    mma_ts(d, ah, dh, idesc, ks > 0);
                    mma_ts(d, ah, dl, idesc, 1);
                    mma_ts(d, al, dh, idesc, 1);
                }
                mma_commit(&br.wdone[s]);
                if (c == 0) mma_commit(&br.qk);  // Q, after K
                if (c == 2) {
                    mma_commit(&br.vdone);
                    // LayerNorm(t) has read the staged rows: the next tile's go
                    // there, queued behind the weights of this tile
                    if (t + 1 < n_my) load_nodes(blockIdx.x + (t + 1) * gridDim.x);
                }
                if (c == kChunks - 1) mma_commit(&br.ofull);
                ++issued;
                progress = true;
            }
            }
            if (progress) {
                idle = 0;
            } else if ((++idle & 63) == 0) {
                // no progress for a while: give up after kWaitNs, or at once
                // when a compute warp's wait already gave up
                const uint64_t tn = now_ns();
                if (idle == 64) idle_since = tn;
                if (flag_set(err) || tn - idle_since > kWaitNs) {
                    atomicExch(err, 1);
                    bail = true;
                    break;
                }
            }
        }
    }
    // every issued MMA complete, every issued bulk copy landed, before exit
    mma_commit(&br.drain);
    mbar_wait(&br.drain, 0, err, false);
    for (int r = issued; r < loaded; ++r) {
        const int s = r % kRing;
        mbar_wait(&br.wfull[s], (ph_wfull >> s) & 1u, err, false);
        ph_wfull ^= 1u << s;
    }
}

// LayerNorm of the tile's node rows (staged in shared memory) into the A
// operand at TMEM column `acol`, by all compute warps: warp (g, k) = (w % 4,
// w / 4) takes columns [24k, 24k + 24) of graph g's rows (thread = row), the
// row statistics are summed over the four column quarters through `red`.
// Writes the row scale exponents and returns after this thread's TMEM stores
// are complete and fenced. `mid` runs between its two barriers (whatever it
// writes is visible to all compute threads after the second), `late` after
// the second.
template <typename Mid, typename Late>
__device__ __forceinline__ void layer_norm(const Params &p, const float *nodes_s, float *red,
                                           int32_t *rscale, const float *gam, const float *bet,
                                           uint32_t tmem, uint32_t acol, int tile, int warp,
                                           int lane, Mid &&mid, Late &&late) {
    const int g = warp & 3, k = warp >> 2, n = lane, N = p.N;
    const bool valid = (int64_t)tile * kGraphs + g < p.B && n < N;
    const int row = 32 * g + n;
    const float4 *xr =
        reinterpret_cast<const float4 *>(nodes_s + (g * N + (valid ? n : 0)) * kNodeStride) + 6 * k;
    float4 x[6];
#pragma unroll
    for (int c = 0; c < 6; ++c) x[c] = xr[c];
    float s1 = 0.f;
#pragma unroll
    for (int c = 0; c < 6; ++c) s1 += (x[c].x + x[c].y) + (x[c].z + x[c].w);
    red[k * 128 + row] = s1;
    named_sync(1, kComputeThreads);
    mid();
    const float mean = ((red[row] + red[128 + row]) + (red[256 + row] + red[384 + row])) / (float)D;
    float v2 = 0.f, dm = 0.f;
#pragma unroll
    for (int c = 0; c < 6; ++c) {
        const float a0 = x[c].x - mean, a1 = x[c].y - mean, a2 = x[c].z - mean, a3 = x[c].w - mean;
        v2 = fmaf(a0, a0, v2);
        v2 = fmaf(a1, a1, v2);
        v2 = fmaf(a2, a2, v2);
        v2 = fmaf(a3, a3, v2);
        dm = fmaxf(dm, fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(a2), fabsf(a3))));
    }
    red[512 + k * 128 + row] = v2;
    red[1024 + k * 128 + row] = dm;
    named_sync(1, kComputeThreads);
    late();
    const float var = ((red[512 + row] + red[640 + row]) + (red[768 + row] + red[896 + row])) / (float)D;
    const float dmax = fmaxf(fmaxf(red[1024 + row], red[1152 + row]), fmaxf(red[1280 + row], red[1408 + row]));
    const float rstd = 1.0f / sqrtf(var + p.ln_eps);
    // an upper bound of |x_n| over the row (gamma, beta maxima follow beta) picks its scale
    const int sr = valid ? scale_exp(dmax * rstd * bet[D] + bet[D + 1]) : 0;
    if (k == 0) rscale[row] = sr;
    const float sc = exp2i(sr);
    uint32_t hi[12], lo[12];
#pragma unroll
    for (int c = 0; c < 6; ++c) {
        const int kk = 24 * k + 4 * c;
        float a[4] = {(x[c].x - mean) * rstd * gam[kk] + bet[kk],
                      (x[c].y - mean) * rstd * gam[kk + 1] + bet[kk + 1],
                      (x[c].z - mean) * rstd * gam[kk + 2] + bet[kk + 2],
                      (x[c].w - mean) * rstd * gam[kk + 3] + bet[kk + 3]};
        if (!valid) a[0] = a[1] = a[2] = a[3] = 0.f;
        split2(a[0] * sc, a[1] * sc, hi[2 * c], lo[2 * c]);
        split2(a[2] * sc, a[3] * sc, hi[2 * c + 1], lo[2 * c + 1]);
    }
    const uint32_t lane_q = (uint32_t)(32 * g) << 16;
#pragma unroll
    for (int c = 0; c < 12; c += 4) {
        tmem_st4(tmem + lane_q + acol + (uint32_t)(12 * k + c), hi + c);
        tmem_st4(tmem + lane_q + acol + kAHalf + (uint32_t)(12 * k + c), lo + c);
    }
    tmem_st_done();
}

__global__ void __launch_bounds__(kThreads, 1) dense_tc_kernel(const Params p) {
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ Barriers br;
    __shared__ uint32_t tmem_slot;
    __shared__ int32_t sw_s[5];
    __shared__ int32_t vmax_s[kGraphs];
    const int N = p.N, NN = N * N, NS = bias_stride(N);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const WsHeader *hd = reinterpret_cast<const WsHeader *>(p.ws);
    int32_t *err = const_cast<int32_t *>(&hd->err);
    float *prm = reinterpret_cast<float *>(sm + Smem::params(N));
    float *w1img = prm, *b1s = w1img + P * P, *w2t = b1s + P, *b2s = w2t + P * H, *gam = b2s + H,
          *bet = gam + D;
    float *red = reinterpret_cast<float *>(sm + Smem::bias);  // LayerNorm statistics (phase C)
    int32_t *rscale = reinterpret_cast<int32_t *>(sm + Smem::rscale(N));
    uint32_t *um_s = reinterpret_cast<uint32_t *>(sm + Smem::umask(N));
    int32_t *rpre_s = reinterpret_cast<int32_t *>(sm + Smem::rpre(N));
    float *bias = reinterpret_cast<float *>(sm + Smem::bias);
    float *nodes_s = reinterpret_cast<float *>(sm + Smem::nodes(N));
    float *stage_base = reinterpret_cast<float *>(sm + Smem::stage(N));

    // ---- set-up: parameters, barriers, TMEM
    {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(p.ws + kWsW1);
        uint32_t *dst = reinterpret_cast<uint32_t *>(w1img);
        for (int i = tid; i < (int)(2 * kW1Half / 4); i += kThreads) dst[i] = src[i];
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // read by the tensor cores
    }
    for (int i = tid; i < P; i += kThreads) b1s[i] = p.b1[i];
    for (int i = tid; i < H * P; i += kThreads) w2t[(i % P) * H + i / P] = p.W2[i];  // [u][h]
    for (int i = tid; i < H; i += kThreads) b2s[i] = p.b2[i];
    for (int i = tid; i < D; i += kThreads) {
        gam[i] = p.ln_w[i];
        bet[i] = p.ln_b[i];
    }
    if (warp == 1) {  // max |gamma|, max |beta| after beta
        float gm = 0.f, bm = 0.f;
        for (int i = lane; i < D; i += 32) {
            gm = fmaxf(gm, fabsf(p.ln_w[i]));
            bm = fmaxf(bm, fabsf(p.ln_b[i]));
        }
        gm = warp_max(gm);
        bm = warp_max(bm);
        if (lane == 0) {
            bet[D] = gm;
            bet[D + 1] = bm;
        }
    }
    if (tid < 5) sw_s[tid] = hd->sw[tid];
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&br.wfull[s], 1);
            mbar_init(&br.wdone[s], 1);
        }
        for (int q = 0; q < 4; ++q) mbar_init(&br.dfull[q], 1);
        mbar_init(&br.nfull, 1);
        mbar_init(&br.xfull, kComputeThreads);
        mbar_init(&br.edone, kComputeThreads);
        mbar_init(&br.qk, 1);
        mbar_init(&br.vdone, 1);
        mbar_init(&br.cfull, kComputeThreads);
        mbar_init(&br.ofull, 1);
        mbar_init(&br.drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = tmem_slot;
    const int n_tiles = (p.B + kGraphs - 1) / kGraphs;
    const int n_my = blockIdx.x < n_tiles ? (n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    if (warp == kComputeWarps) {
        if (lane == 0) control_loop(p, sm, br, tmem, n_my, nodes_s, err);
        __syncwarp();
    } else {
        const int g = warp & 3, h = warp >> 2, n = lane;  // graph (lane quarter), head, node
        const uint32_t lane_q = (uint32_t)(32 * g) << 16;
        const float qk_scale = kLog2e / sqrtf((float)DH);  // scores in log2 units
        const int quad = warp >> 2;                         // relation-MLP blocks quad, quad + 4, ...
        uint32_t ph_qk = 0, ph_v = 0, ph_of = 0;

        // Relation-MLP pairs: only the unmasked ones. A masked pair's logit is
        // -inf whatever its relation MLP gives, so its features are never read;
        // the unmasked pairs of a tile are numbered in (graph, query, key)
        // order and taken in 128-pair blocks.
        // mask_copy(tl): tile tl's mask values into the staging region above
        // the prefetch slots and the attention's staging (cp.async, issued
        // during the previous tile's attention); mask_words(tl), once the
        // copies are complete and visible: the unmasked-key words (four
        // threads per (graph, row)); mask_scan(): their row prefix (warp 0;
        // visible after the next barrier)
        float *mask_s = stage_base + Smem::mask_off(N);
        auto mask_copy = [&](int tl) {
            const int64_t g0 = (int64_t)tl * kGraphs;
            const int np = (int)((p.B - g0 < kGraphs ? p.B - g0 : kGraphs) * NN);
            for (int pi = tid; pi < np; pi += kComputeThreads)
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(mask_s + pi)),
                             "l"(p.mask + g0 * NN + pi)
                             : "memory");
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        auto mask_words = [&](int tl) {
            {
                // word r = tid / 4 (graph r / 32, row r % 32), keys
                // [6 (tid % 4), 6 (tid % 4) + 6) from this thread, OR-ed over the 4
                const int r = tid >> 2, part = tid & 3, gg = r >> 5, nn = r & 31;
                uint32_t w = 0;
                if (nn < N && (int64_t)tl * kGraphs + gg < p.B) {
                    const float *mr = mask_s + gg * NN + nn * N;
#pragma unroll
                    for (int k = 0; k < kMaxN / 4; ++k) {
                        const int j = (kMaxN / 4) * part + k;
                        if (j < N) w |= (mr[j] < 0.5f ? 0u : 1u) << j;
                    }
                }
                w |= __shfl_xor_sync(kFull, w, 1);
                w |= __shfl_xor_sync(kFull, w, 2);
                if (part == 0) um_s[r] = w;
            }
        };
        auto mask_scan = [&]() {
            if (warp == 0) {
                int cr[4], sum = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    cr[k] = __popc(um_s[4 * lane + k]);
                    sum += cr[k];
                }
                int incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += y;
                }
                int ex = incl - sum;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    rpre_s[4 * lane + k] = ex;
                    ex += cr[k];
                }
                if (lane == 31) rpre_s[128] = incl;
            }
        };
        // the idx-th unmasked pair of the tile (idx < its count): the row by a
        // binary search of the prefix, the key as that row's k-th unmasked bit
        auto pair_of = [&](int idx) -> int {
            int r = 0;
#pragma unroll
            for (int st = 64; st > 0; st >>= 1)
                if (rpre_s[r + st] <= idx) r += st;
            const int j = (int)__fns(um_s[r], 0, idx - rpre_s[r] + 1);
            return (r >> 5) * NN + (r & 31) * N + j;
        };
        // relation-MLP prefetch slots: thread T's 16 features at float4
        // 4 T + (c ^ (T / 2 % 4)) for quarter c (the swizzle keeps a warp's
        // reads of one quarter and its copies of eight whole pairs free of
        // bank conflicts)
        float4 *slots = reinterpret_cast<float4 *>(stage_base);
        const int swz = (tid >> 1) & 3;
        const float4 *pslot = slots + 4 * tid;
        // this thread's pair in block blk of the current words, or -1
        auto pair_at = [&](int blk) -> int {
            const int idx = 128 * blk + 32 * g + lane;
            return idx < rpre_s[128] ? pair_of(idx) : -1;
        };
        // block blk of tile tl (warp-uniform call; pi = this thread's pair in
        // it): the warp copies its own 32 pairs, four lanes per pair (lane % 4 =
        // the quarter), eight pairs per copy instruction, so that consecutive
        // pairs give 512 consecutive bytes
        auto fetch_pairs = [&](int tl, int pi) {
            const float *src = p.pair + (int64_t)tl * kGraphs * NN * P + 4 * (lane & 3);
            __syncwarp();  // every lane has read its slot (block blk - 4)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int sl = 8 * j + (lane >> 2);
                const int pj = __shfl_sync(kFull, pi, sl);
                const int dt = 32 * warp + sl;
                if (pj >= 0)
                    cp_async16(smem_u32(slots + 4 * dt + ((lane & 3) ^ ((dt >> 1) & 3))),
                               src + (int64_t)pj * P);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };

        // prologue: the first tile's unmasked-pair words, its LayerNorm with
        // their prefix and its first relation-MLP blocks' prefetch
        // (the pair of the quad's second block is found here too, beside the
        // first's search; both are kept for the relation MLP: the second
        // block's prefetch and the two blocks' bias writes)
        int pi_first = -1, pi_second = -1;
        auto first_fetch = [&](int tl) {  // (always one commit group)
            pi_first = pair_at(quad);
            pi_second = pair_at(quad + 4);
            if (128 * quad < rpre_s[128])
                fetch_pairs(tl, pi_first);
            else
                asm volatile("cp.async.commit_group;" ::: "memory");
        };
        // The epilogue works per graph: its output block ([N][D], contiguous in
        // global memory) is staged in shared memory, starting as the residual
        // rows (copied in during the next tile's LayerNorm, one commit group);
        // the four head warps of graph g add the out-projection there, then
        // the same 128 threads write it as consecutive float4s (gt + 128 k).
        const int gt = 32 * h + lane;
        auto res_copy = [&](int tl) {
            const int64_t bg = (int64_t)tl * kGraphs + g;
            if (bg < p.B) {
                const float4 *xg = reinterpret_cast<const float4 *>(p.nodes + bg * N * (int64_t)D);
                float *os = stage_base + Smem::out_off + g * N * kOutStride;
#pragma unroll
                for (int k = 0; k < kOutVec; ++k) {
                    const int f = gt + 128 * k;
                    if (f < N * D / 4) {
                        const int row = f / (D / 4), c4 = f - row * (D / 4);
                        cp_async16(smem_u32(os + row * kOutStride + 4 * c4), xg + f);
                    }
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        if (n_my > 0) {
            mask_copy(blockIdx.x);
            asm volatile("cp.async.wait_all;" ::: "memory");
            named_sync(1, kComputeThreads);
            mask_words(blockIdx.x);
            mbar_wait(&br.nfull, 0, err);  // the first tile's node rows
            layer_norm(p, nodes_s, red, rscale, gam, bet, tmem, col_a(0), blockIdx.x, warp, lane,
                       mask_scan, [&] { first_fetch(blockIdx.x); });
            mbar_arrive(&br.xfull);
            named_sync(1, kComputeThreads);  // LayerNorm statistics read, the bias region is free
        }
        uint32_t ph_ed = 0, ph_df = 0;

        for (int it = 0; it < n_my; ++it) {
            const int tile = blockIdx.x + it * gridDim.x;
            const uint32_t acol = col_a(it);
            const int64_t b = (int64_t)tile * kGraphs + g;
            const bool rvalid = b < p.B && n < N;
            if (tid < kGraphs) vmax_s[tid] = 0;

            // ======== phase A: relation MLP, thread = pair 32 g + n of 128-pair blocks
            // quad, quad + 4, ...: the first layer on the tensor cores (the pair's
            // features, scaled and split, are the A operand in this quad's TMEM slot;
            // the quad's first thread issues its MMAs). Software-pipelined: block i's
            // hidden values are read back, block i + 1 is split and issued, then block
            // i's epilogue runs while the tensor cores work.
            bool guard = it > 0;  // the last LayerNorm's statistics share the bias region
            const int npairs = rpre_s[128];            // the tile's unmasked pairs
            const int nblk = (npairs + 127) >> 7;       // in 128-pair blocks
            const uint32_t slot_col = mlp_col(it, quad);
            const uint32_t mslot_t = tmem + lane_q + slot_col;
            const bool issuer = (warp & 3) == 0 && lane == 0;
            auto split_issue = [&](int blk, int &sp) {
                const bool valid = 128 * blk + 32 * g + lane < npairs;
                asm volatile("cp.async.wait_all;" ::: "memory");
                __syncwarp();  // the slots are filled by other lanes' copies
                float pf[P];
#pragma unroll
                for (int c = 0; c < P / 4; ++c) {
                    const float4 v = valid ? pslot[c ^ swz] : make_float4(0.f, 0.f, 0.f, 0.f);
                    pf[4 * c] = v.x;
                    pf[4 * c + 1] = v.y;
                    pf[4 * c + 2] = v.z;
                    pf[4 * c + 3] = v.w;
                }
                if (blk + 4 < nblk) fetch_pairs(tile, blk == quad ? pi_second : pair_at(blk + 4));
                float mx = 0.f;
#pragma unroll
                for (int u = 0; u < P; ++u) mx = fmaxf(mx, fabsf(pf[u]));
                sp = scale_exp(mx);
                const float sc = exp2i(sp);
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) split2(pf[2 * c] * sc, pf[2 * c + 1] * sc, hi[c], lo[c]);
                tmem_st8(mslot_t, hi);
                tmem_st8(mslot_t + 8, lo);
                tmem_st_done();
                named_sync(2 + quad, 128);  // the block's 128 rows are in TMEM
                if (issuer) {
                    fence_after();
                    const uint32_t base = tmem + slot_col;
                    constexpr uint32_t idesc_m = idesc_f16(P, 128);
                    const uint32_t w1h = smem_u32(w1img);
                    const uint64_t w1dh = smem_desc(w1h, 128, 256);
                    const uint64_t w1dl = smem_desc(w1h + kW1Half, 128, 256);
                    mma_ts(base + 16, base, w1dh, idesc_m, 0);
                    mma_ts(base + 16, base, w1dl, idesc_m, 1);
                    mma_ts(base + 16, base + 8, w1dh, idesc_m, 1);
                    mma_commit(&br.dfull[quad]);
                }
            };
            int sp = 0;
            if (quad < nblk) split_issue(quad, sp);
            for (int blk = quad; blk < nblk; blk += 4) {
                const int idx = 128 * blk + 32 * g + lane;
                const bool valid = idx < npairs;
                mbar_wait(&br.dfull[quad], ph_df, err);
                ph_df ^= 1u;
                fence_after();
                float hid[P];
                tmem_ld16(mslot_t + 16, hid);
                const float unsc = exp2i(-sp) * exp2i(-sw_s[4]);
                if (blk + 4 < nblk) split_issue(blk + 4, sp);
                // b1, SiLU, then r = W2 silu + b2 as head pairs (0, 1), (2, 3)
                float2 r01 = make_float2(b2s[0], b2s[1]), r23 = make_float2(b2s[2], b2s[3]);
#pragma unroll
                for (int u4 = 0; u4 < P / 4; ++u4) {
                    const float4 bq = reinterpret_cast<const float4 *>(b1s)[u4];
                    const float bb[4] = {bq.x, bq.y, bq.z, bq.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int u = 4 * u4 + i;
                        const float a = fmaf(hid[u], unsc, bb[i]);
                        const float sl = __fdividef(a, 1.0f + __expf(-a));
                        const float2 ss = make_float2(sl, sl);
                        const float4 w = reinterpret_cast<const float4 *>(w2t)[u];
                        r01 = ffma2(make_float2(w.x, w.y), ss, r01);
                        r23 = ffma2(make_float2(w.z, w.w), ss, r23);
                    }
                }
                if (guard) {  // every thread is past that LayerNorm once tile it-1 is done
                    mbar_wait(&br.edone, ph_ed, err);
                    ph_ed ^= 1u;
                    guard = false;
                }
                if (valid) {
                    const int pi = blk == quad ? pi_first : (blk == quad + 4 ? pi_second : pair_of(idx));
                    const int gg = pi / NN, rem = pi - gg * NN, nn = rem / N, j = rem - nn * N;
                    float *bw = bias + (gg * H * N + j) * NS + nn;  // head stride N * NS
                    bw[0] = r01.x * kLog2e;
                    bw[N * NS] = r01.y * kLog2e;
                    bw[2 * N * NS] = r23.x * kLog2e;
                    bw[3 * N * NS] = r23.y * kLog2e;
                }
            }
            if (guard) {  // this thread had no block: the barrier phase is still consumed
                mbar_wait(&br.edone, ph_ed, err);
                ph_ed ^= 1u;
                guard = false;
            }
            named_sync(1, kComputeThreads);  // every unmasked pair's bias written
            mbar_wait(&br.qk, ph_qk, err);  // Q and K (V is waited for before its use)
            ph_qk ^= 1u;
            fence_after();
            // the next tile's mask values (its LayerNorm reads them)
            if (it + 1 < n_my) mask_copy(tile + gridDim.x);

            // ======== phase B: attention of head h in graph g, thread = query node n
            const int sr = rscale[32 * g + n];
            // the normalised context in the MMA accumulator layout: rows
            // 16 m + tq + 8 i, dims 8 t + 2 tr + j at [m][t][2 i + j]
            float cctx[2][3][4];
            const int tq = lane >> 2, tr = lane & 3;
            {
                // The warp's staging: after the softmax the V rows (the B
                // operand of the context product).
                float *sv = stage_base + warp * Smem::warp_stage(N);
                const float uv = exp2i(-sr) * exp2i(-sw_s[2]);
                const int nq = b < p.B ? N : 0;  // the graph's rows (queries) and keys
                // Warp-level tensor-core MMAs (m16n8k16, f16 operands split into a
                // rounded part and its remainder, three products per term as the
                // projections' split does, each operand row scaled by a power of
                // two into [2^12, 2^13) for the split): 32 query rows (2 row
                // tiles) x 24 keys (3 tiles of 8), then x 24 dims. Fragment
                // coordinates: row group tq, column pair tr.
                // the row owner's ranges of its Q and K rows over the head's dims
                int sq_n, sk_n;
                {
                    float mq = 0.f, mk = 0.f;
#pragma unroll
                    for (int c0 = 0; c0 < DH; c0 += 8) {
                        float v[8];
                        tmem_ld8(tmem + lane_q + (uint32_t)(h * DH + c0), v);
#pragma unroll
                        for (int i = 0; i < 8; ++i) mq = fmaxf(mq, fabsf(v[i]));
                        tmem_ld8(tmem + lane_q + (uint32_t)(D + h * DH + c0), v);
#pragma unroll
                        for (int i = 0; i < 8; ++i) mk = fmaxf(mk, fabsf(v[i]));
                    }
                    sq_n = scale_exp(mq);
                    sk_n = scale_exp(mk);
                }
                // fragment scales: rows 16 m + 8 i + tq, keys 8 t + tq
                float aq[2][2], bk[3];
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int i = 0; i < 2; ++i) aq[m][i] = exp2i(__shfl_sync(kFull, sq_n, 16 * m + 8 * i + tq));
#pragma unroll
                for (int t = 0; t < 3; ++t) bk[t] = exp2i(__shfl_sync(kFull, sk_n, 8 * t + tq));
                float sacc[2][3][4];
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int t = 0; t < 3; ++t)
#pragma unroll
                        for (int e = 0; e < 4; ++e) sacc[m][t][e] = 0.f;
                // scores S = Q K^T, k over the head's dims in 2 steps of 16 (the
                // second half zero). The fragments come straight from TMEM
                // (16x256b loads: lane (tq, tr) holds rows tq, tq + 8 of a
                // 16-row half at columns 2 tr, 2 tr + 1 of an 8-column chunk).
                // Padding rows and keys hold exact zeros (their LayerNorm rows
                // are zero); their scores are masked or never stored.
#pragma unroll
                for (int st = 0; st < 2; ++st) {
                    const uint32_t cq = (uint32_t)(h * DH + 16 * st), ck = cq + (uint32_t)D;
                    // keys: chunks 0 (dims 0-7 of the step) and 1 (8-15; unused in
                    // the second step) of both 16-row halves
                    uint32_t k00[4], k10[4], k01[4], k11[4];
                    tmem_ld16x8(tmem + lane_q + ck, k00);
                    tmem_ld16x8(tmem + lane_q + (16u << 16) + ck, k10);
                    tmem_ld16x8(tmem + lane_q + ck + 8u, k01);
                    tmem_ld16x8(tmem + lane_q + (16u << 16) + ck + 8u, k11);
                    tmem_wait_tied(k00, k10, k01, k11);
                    uint32_t bh[3][2], bl[3][2];
#pragma unroll
                    for (int t = 0; t < 3; ++t) {
                        // key tile t: rows tq / tq + 8 of the first half, rows tq of the second
                        const uint32_t *c0 = t < 2 ? k00 : k10, *c1 = t < 2 ? k01 : k11;
                        const int o = t == 1 ? 2 : 0;
                        split2(__uint_as_float(c0[o]) * bk[t], __uint_as_float(c0[o + 1]) * bk[t], bh[t][0], bl[t][0]);
                        if (st == 0) {
                            split2(__uint_as_float(c1[o]) * bk[t], __uint_as_float(c1[o + 1]) * bk[t], bh[t][1], bl[t][1]);
                        } else {
                            bh[t][1] = bl[t][1] = 0u;
                        }
                    }
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        uint32_t q0[4], q1[4];
                        tmem_ld16x8(tmem + lane_q + ((uint32_t)(16 * m) << 16) + cq, q0);
                        tmem_ld16x8(tmem + lane_q + ((uint32_t)(16 * m) << 16) + cq + 8u, q1);
                        tmem_wait_tied(q0, q1);
                        uint32_t ah[4], al[4];
                        split2(__uint_as_float(q0[0]) * aq[m][0], __uint_as_float(q0[1]) * aq[m][0], ah[0], al[0]);
                        split2(__uint_as_float(q0[2]) * aq[m][1], __uint_as_float(q0[3]) * aq[m][1], ah[1], al[1]);
                        if (st == 0) {
                            split2(__uint_as_float(q1[0]) * aq[m][0], __uint_as_float(q1[1]) * aq[m][0], ah[2], al[2]);
                            split2(__uint_as_float(q1[2]) * aq[m][1], __uint_as_float(q1[3]) * aq[m][1], ah[3], al[3]);
                        } else {
                            ah[2] = ah[3] = al[2] = al[3] = 0u;
                        }
#pragma unroll
                        for (int t = 0; t < 3; ++t) {
                            mma_f16(sacc[m][t], al, bh[t]);
                            mma_f16(sacc[m][t], ah, bl[t]);
                            mma_f16(sacc[m][t], ah, bh[t]);
                        }
                    }
                }
                // back to log2 units: row r, key c by 2^-(sq_r + sk_c) times the
                // projections' unscaling (and 1 / sqrt(head_dim) log2 e for Q)
                {
                    const float fq_n = exp2i(-sq_n) * exp2i(-sr) * exp2i(-sw_s[0]) * qk_scale;
                    const float fk_n = exp2i(-sk_n) * exp2i(-sr) * exp2i(-sw_s[1]);
                    float fq[2][2], fk[3][2];
#pragma unroll
                    for (int m = 0; m < 2; ++m)
#pragma unroll
                        for (int i = 0; i < 2; ++i) fq[m][i] = __shfl_sync(kFull, fq_n, 16 * m + 8 * i + tq);
#pragma unroll
                    for (int t = 0; t < 3; ++t)
#pragma unroll
                        for (int j = 0; j < 2; ++j) fk[t][j] = __shfl_sync(kFull, fk_n, 8 * t + 2 * tr + j);
#pragma unroll
                    for (int m = 0; m < 2; ++m)
#pragma unroll
                        for (int t = 0; t < 3; ++t)
#pragma unroll
                            for (int e = 0; e < 4; ++e) sacc[m][t][e] *= fq[m][e >> 1] * fk[t][e & 1];
                }
                // bias (log2 units) on the query's unmasked keys, -inf on the
                // others and on keys past the graph's nodes; then the row softmax
                // over the quad of lanes sharing a row (an all -inf row gives NaN,
                // as the reference)
                const float *bh = bias + (g * H + h) * N * NS;
                float zr[2][2];
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int row = 16 * m + tq + 8 * i;
                        const bool rv = row < nq;
                        const uint32_t wr = rv ? um_s[32 * g + row] : 0xffffffffu;
                        float mx = -INFINITY;
#pragma unroll
                        for (int t = 0; t < 3; ++t)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int key = 8 * t + 2 * tr + e;
                                const bool live = key < nq && ((wr >> key) & 1u);
                                const float bv = live ? (rv ? bh[key * NS + row] : 0.f) : -INFINITY;
                                const float sv2 = sacc[m][t][2 * i + e] + bv;
                                sacc[m][t][2 * i + e] = sv2;
                                mx = fmaxf(mx, sv2);
                            }
                        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
                        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
                        float z = 0.f;
#pragma unroll
                        for (int t = 0; t < 3; ++t)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float pe = ex2(sacc[m][t][2 * i + e] - mx);
                                sacc[m][t][2 * i + e] = pe;
                                z += pe;
                            }
                        z += __shfl_xor_sync(kFull, z, 1);
                        z += __shfl_xor_sync(kFull, z, 2);
                        zr[m][i] = z;
                    }
                // the V rows (scaled) into the warp's staging, and the graph's
                // largest |V|
                mbar_wait(&br.vdone, ph_v, err);
                ph_v ^= 1u;
                fence_after();
                float vm = 0.f;
#pragma unroll
                for (int c0 = 0; c0 < DH; c0 += 8) {
                    float vf[8];
                    tmem_ld8(tmem + lane_q + (uint32_t)(2 * D + h * DH + c0), vf);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        vf[i] *= uv;
                        vm = fmaxf(vm, fabsf(vf[i]));
                    }
                    if (rvalid) {
                        *reinterpret_cast<float4 *>(sv + n * DH + c0) = make_float4(vf[0], vf[1], vf[2], vf[3]);
                        *reinterpret_cast<float4 *>(sv + n * DH + c0 + 4) = make_float4(vf[4], vf[5], vf[6], vf[7]);
                    }
                }
                vm = rvalid ? vm : 0.f;
                vm = warp_max(vm);
                if (lane == 0) atomicMax(&vmax_s[g], __float_as_int(vm));
                // context = P V on f16 MMAs (m16n8k16), each operand split into
                // a rounded f16 part and its remainder as the projections' split
                // does, three products per term; P scaled by 2^12 (P <= 1), V by
                // this warp's 2^sv (its largest |V| to [2^12, 2^13)), both exact;
                // k over the keys in 2 steps of 16 (the second half zero). P's
                // accumulator fragment is its A fragment as it stands: keys
                // 8 t + 2 tr, + 1 are registers (0, 1) of row tq and (2, 3) of
                // row tq + 8.
                const int sv_e = scale_exp(vm);
                const float vsc = exp2i(sv_e), psc = 4096.f;
                float cacc[2][3][4];
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int t = 0; t < 3; ++t)
#pragma unroll
                        for (int e = 0; e < 4; ++e) cacc[m][t][e] = 0.f;
#pragma unroll
                for (int st = 0; st < 2; ++st) {
                    uint32_t ah[2][4], al[2][4];
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        split2(sacc[m][2 * st][0] * psc, sacc[m][2 * st][1] * psc, ah[m][0], al[m][0]);
                        split2(sacc[m][2 * st][2] * psc, sacc[m][2 * st][3] * psc, ah[m][1], al[m][1]);
                        if (st == 0) {
                            split2(sacc[m][1][0] * psc, sacc[m][1][1] * psc, ah[m][2], al[m][2]);
                            split2(sacc[m][1][2] * psc, sacc[m][1][3] * psc, ah[m][3], al[m][3]);
                        } else {
                            ah[m][2] = ah[m][3] = al[m][2] = al[m][3] = 0u;
                        }
                    }
                    const int k0 = 16 * st + 2 * tr;  // keys k0, k0 + 1, then k0 + 8, k0 + 9
#pragma unroll
                    for (int t = 0; t < DH / 8; ++t) {
                        const int dim = 8 * t + tq;
                        const float v0 = k0 < nq ? sv[k0 * DH + dim] : 0.f;
                        const float v1 = k0 + 1 < nq ? sv[(k0 + 1) * DH + dim] : 0.f;
                        const float v2 = st == 0 && k0 + 8 < nq ? sv[(k0 + 8) * DH + dim] : 0.f;
                        const float v3 = st == 0 && k0 + 9 < nq ? sv[(k0 + 9) * DH + dim] : 0.f;
                        uint32_t bh[2], bl[2];
                        split2(v0 * vsc, v1 * vsc, bh[0], bl[0]);
                        split2(v2 * vsc, v3 * vsc, bh[1], bl[1]);
#pragma unroll
                        for (int m = 0; m < 2; ++m) {
                            mma_f16(cacc[m][t], al[m], bh);
                            mma_f16(cacc[m][t], ah[m], bl);
                            mma_f16(cacc[m][t], ah[m], bh);
                        }
                    }
                }
                // normalised (rows past the graph's nodes: zero)
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int row = 16 * m + tq + 8 * i;
                        const float inv = row < nq ? exp2i(-12) * exp2i(-sv_e) * (1.0f / zr[m][i]) : 0.f;
#pragma unroll
                        for (int t = 0; t < DH / 8; ++t)
#pragma unroll
                            for (int j = 0; j < 2; ++j)
                                cctx[m][t][2 * i + j] = row < nq ? cacc[m][t][2 * i + j] * inv : 0.f;
                    }
            }
            asm volatile("cp.async.wait_all;" ::: "memory");  // the next tile's mask values
            named_sync(1, kComputeThreads);  // every graph's largest |V| known; staging free
            // the next tile's unmasked-pair words (this tile's are read)
            if (it + 1 < n_my) mask_words(tile + gridDim.x);
            // the context (|ctx| <= max |V| of the graph) as the out-projection's A
            // operand, stored from the accumulator layout (16x128b: dims
            // 8 t + 2 tr, + 1 are packed column h DH / 2 + 4 t + tr of rows tq,
            // tq + 8 of each 16-row half)
            const int sc_g = scale_exp(__int_as_float(vmax_s[g]));
            {
                const float sc = exp2i(sc_g);
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int t = 0; t < DH / 8; ++t) {
                        uint32_t h0, l0, h1, l1;
                        split2(cctx[m][t][0] * sc, cctx[m][t][1] * sc, h0, l0);
                        split2(cctx[m][t][2] * sc, cctx[m][t][3] * sc, h1, l1);
                        const uint32_t a = tmem + lane_q + ((uint32_t)(16 * m) << 16) + acol +
                                           (uint32_t)(h * DH / 2 + 4 * t);
                        tmem_st16x4(a, h0, h1);
                        tmem_st16x4(a + kAHalf, l0, l1);
                    }
            }
            tmem_st_done();
            mbar_arrive(&br.cfull);

            // ======== phase C: LayerNorm of the next tile, then out-projection + residual
            if (it + 1 < n_my) {
                mbar_wait(&br.nfull, (uint32_t)(it + 1) & 1u, err);  // the next tile's node rows
                // with the prefix of the next tile's unmasked-pair words, and the
                // prefetch of its first relation-MLP blocks
                // (the residual copies go in after the next tile's prefetch, which
                // is needed first; every thread has read the mask values in the
                // staging region by then)
                layer_norm(p, nodes_s, red, rscale, gam, bet, tmem, col_a(it + 1),
                           tile + gridDim.x, warp, lane, mask_scan,
                           [&] {
                               first_fetch(tile + gridDim.x);
                               res_copy(tile);
                           });
                mbar_arrive(&br.xfull);
            } else {
                res_copy(tile);
            }
            const bool failed = flag_set(err);
            const bool o_ok = mbar_wait(&br.ofull, ph_of, err);
            ph_of ^= 1u;
            fence_after();
            {
                const float uo = exp2i(-sc_g) * exp2i(-sw_s[3]);
                float *os = stage_base + Smem::out_off + g * N * kOutStride;
                // this thread's residual copies (committed last), then the whole
                // graph's
                asm volatile("cp.async.wait_group 0;" ::: "memory");
                named_sync(6 + g, 128);
#pragma unroll
                for (int c0 = 0; c0 < DH; c0 += 8) {
                    float v[8];
                    tmem_ld8(tmem + lane_q + (uint32_t)(h * DH + c0), v);
                    if (n < N) {
                        float4 *w = reinterpret_cast<float4 *>(os + n * kOutStride + h * DH + c0);
                        const float4 x0 = w[0], x1 = w[1];
                        w[0] = make_float4(fmaf(v[0], uo, x0.x), fmaf(v[1], uo, x0.y),
                                           fmaf(v[2], uo, x0.z), fmaf(v[3], uo, x0.w));
                        w[1] = make_float4(fmaf(v[4], uo, x1.x), fmaf(v[5], uo, x1.y),
                                           fmaf(v[6], uo, x1.z), fmaf(v[7], uo, x1.w));
                    }
                }
                fence_before();
                mbar_arrive(&br.edone);  // this thread no longer reads columns [0, 288)
                named_sync(6 + g, 128);  // graph g's output block complete
                const float fail = failed || !o_ok ? NAN : 0.f;
                float4 *og = reinterpret_cast<float4 *>(p.out + b * N * (int64_t)D);
                const int nf4 = N * D / 4;
#pragma unroll
                for (int k = 0; k < kOutVec; ++k) {
                    const int f = gt + 128 * k;
                    if (b < p.B && f < nf4) {
                        const int row = f / (D / 4), c4 = f - row * (D / 4);
                        const float4 v = *reinterpret_cast<const float4 *>(os + row * kOutStride + 4 * c4);
                        og[f] = make_float4(v.x + fail, v.y + fail, v.z + fail, v.w + fail);
                    }
                }
            }
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
}

}  // namespace tc

// Host side. dense_block_tc_shape: whether (N, D, H, P) is this kernel's shape.
bool dense_block_tc_shape(int32_t N, int32_t D, int32_t H, int32_t P) {
    return P == tc::P && H == tc::H && D == tc::D && N >= 1 && N <= tc::kMaxN &&
           tc::Smem::total(N) <= 227u * 1024u;
}

size_t dense_block_tc_workspace() { return tc::kWsBytes; }

// The block on the tensor cores (the caller checked the shape).
gat_status_t dense_block_tc(int32_t B, int32_t N, int32_t D, int32_t H, int32_t P,
                            const float *nodes, const float *pair, const float *mask,
                            const float *ln_w, const float *ln_b, float ln_eps, const float *Wq,
                            const float *Wk, const float *Wv, const float *W1, const float *b1,
                            const float *W2, const float *b2, const float *Wout, float *out,
                            void *workspace, size_t workspace_bytes, cudaStream_t s) {
    if (!dense_block_tc_shape(N, D, H, P)) return GAT_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < tc::kWsBytes || !aligned16(workspace))
        return fail(GAT_ERR_WORKSPACE,
                    "gat_dense_masked_attention: this shape needs a 16-byte aligned workspace of "
                    "%zu bytes (got %zu)", tc::kWsBytes, workspace_bytes);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    tc::dense_prep_kernel<<<5, tc::kPrepThreads, 0, s>>>(Wq, Wk, Wv, Wout, W1, ws);
    gat_status_t st = check_launch("gat_dense_masked_attention (weight prep)");
    if (st != GAT_OK) return st;
    const uint32_t smem = tc::Smem::total(N);
    static std::atomic<int> smem_set[kMaxDevices];
    cudaError_t e = allow_dynamic_smem(smem_set, tc::dense_tc_kernel, (int)tc::Smem::total(tc::kMaxN));
    if (e != cudaSuccess) return cuda_fail(e, "gat_dense_masked_attention: smem attribute");
    tc::Params p{B, N, nodes, pair, mask, ln_w, ln_b, ln_eps, W1, b1, W2, b2, ws, out};
    const int64_t tiles = (B + tc::kGraphs - 1) / tc::kGraphs;
    int64_t blocks = sm_count();
    if (blocks > tiles) blocks = tiles;
    tc::dense_tc_kernel<<<(unsigned)blocks, tc::kThreads, smem, s>>>(p);
    return check_launch("gat_dense_masked_attention (tcgen05)");
}

// Error flag of the last call that used `workspace` (synchronises `stream`).
gat_status_t dense_block_tc_status(const void *workspace, cudaStream_t s) {
    int32_t flag = 0;
    const tc::WsHeader *hd = static_cast<const tc::WsHeader *>(workspace);
    cudaError_t e = cudaMemcpyAsync(&flag, &hd->err, sizeof(flag), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "gat_dense_masked_attention_status");
    if (flag)
        return fail(GAT_ERR_CUDA, "gat_dense_masked_attention: a bounded wait on the tensor-core "
                    "pipeline gave up; that call's outputs were written as NaN");
    return GAT_OK;
}

}  // namespace gat
