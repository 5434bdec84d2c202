// dense_block_tc.cu - the dense-masked attention block of the block page's
// module shape (Kimi-K2.6 l2_p4, reference model: P = 16 pair features,
// H = 4 heads of 24 dims, D = 96, up to 24 nodes) with its contractions on the
// 5th-generation tensor cores (tcgen05, kind::f16, fp32 accumulators in TMEM).
//
// Precision: fp32 results from fp16 tensor-core products. Every operand row
// (a node row, a pair's features, a weight matrix) is scaled by a power of
// two 2^s that brings its largest magnitude into [2^12, 2^13), then split
// x 2^s = hi + lo with hi = fp16(x 2^s) and lo = fp16(x 2^s - hi) (both round
// to nearest even). A B ~ hi_A hi_B + hi_A lo_B + lo_A hi_B: the dropped
// lo_A lo_B and lo's own rounding are ~2^-22 of the row's largest term, the
// fp32 accumulation of the products is exact per product, and the scales are
// undone exactly in fp32 afterwards. Three fp16 MMAs cost what 1.5 tf32 MMAs
// do, for the same accuracy as the 3xTF32 split.
//
// Every A operand lives in TMEM (written by tcgen05.st from the registers of
// the thread owning the row), so the tensor cores read only the weights from
// shared memory. A tile is 4 graphs padded to 32 rows: graph g owns TMEM lanes
// 32g..32g+31, which warps g, g+4, g+8, g+12 may access.
//
// 17 warps per CTA, one CTA per SM, persistent over tiles:
//   warp 16 (control; its lane 0): streams the pre-split weight chunks
//       (Q0 Q1 K0 K1 V0 V1 O0 O1, 48 rows each) through a 4-slot shared
//       memory ring with bulk copies, issues every MMA and commits each group
//       to the mbarrier its consumer waits on;
//   quad 0 (warps 0-3): LayerNorm, one thread per node row, from node rows
//       staged in shared memory by cp.async (the next tile's rows are fetched
//       as soon as this tile's are normalised) -> A operand in TMEM;
//   all quads: the relation MLP, one thread per node pair: the pair's 16
//       features go to its TMEM lane as the A operand of W1 (M = 128 pairs,
//       N = 16, K = 16), the same thread reads the 16 hidden values back,
//       applies b1, SiLU, W2, b2 and the edge mask (-inf where masked) and
//       writes the bias of all heads to shared memory;
//   warp (g, h) = (w % 4, w / 4): attention of head h in graph g, one thread
//       per query node: Q row from TMEM, K and V rows staged in shared memory,
//       scores + bias, two-pass softmax, context; the context becomes the A
//       operand of the out-projection (scaled per graph by the largest |V|,
//       which bounds it);
//   epilogue: out-projection columns [24h, 24h + 24) + residual.
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
constexpr int kNB = 48;                           // weight chunk rows (MMA N)
constexpr int kChunks = 8;                        // Q0 Q1 K0 K1 V0 V1 O0 O1
constexpr int kQkvChunks = 6;
constexpr int kRing = 4;
constexpr uint32_t kChunkHalf = kNB * D * 2;      // one of hi / lo, fp16
constexpr uint32_t kChunkBytes = 2 * kChunkHalf;
constexpr uint32_t kW1Half = P * P * 2;
constexpr int kNodeStride = 100;                  // floats per staged node row
// TMEM columns (32-bit each): fp32 accumulators, or fp16 pairs for A operands
constexpr uint32_t kColAhi = 288, kColAlo = 336;  // A operand (x_n, then the context), K = 96
constexpr uint32_t kColMlp = 384;                 // 4 slots of A hi (8) | A lo (8) | D (16)
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 1000000000ull;       // a wait gives up after 1 s (never expected)

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

// ---------------------------------------------------------------------------
// prep: weights -> scaled fp16 hi / lo images in the shared-memory layout
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 256;

// Block b < 8: rows [48 (b % 2), +48) of Wq, Wk, Wv, Wout (b / 2); block 8: W1.
__global__ void __launch_bounds__(kPrepThreads)
dense_prep_kernel(const float *__restrict__ Wq, const float *__restrict__ Wk,
                  const float *__restrict__ Wv, const float *__restrict__ Wout,
                  const float *__restrict__ W1, unsigned char *__restrict__ ws) {
    __shared__ float red[kPrepThreads / 32];
    const int b = blockIdx.x, tid = threadIdx.x;
    const int which = b < 8 ? b / 2 : 4;
    const float *W = which == 0 ? Wq : which == 1 ? Wk : which == 2 ? Wv : which == 3 ? Wout : W1;
    const int K = b < 8 ? D : P, rows = b < 8 ? kNB : P, row0 = b < 8 ? (b % 2) * kNB : 0;
    const int n_all = K * K;
    float m = 0.f;
    for (int i = tid; i < n_all; i += kPrepThreads) m = fmaxf(m, fabsf(__ldg(W + i)));
    m = warp_max(m);
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    m = 0.f;
#pragma unroll
    for (int w = 0; w < kPrepThreads / 32; ++w) m = fmaxf(m, red[w]);
    const int s = scale_exp(m);
    WsHeader *hd = reinterpret_cast<WsHeader *>(ws);
    if (tid == 0) {
        if (b == 8 || b % 2 == 0) hd->sw[which] = s;
        if (b == 0) hd->err = 0;
    }
    const float sc = exp2i(s);
    unsigned char *dst = ws + (b < 8 ? kWsChunks + (size_t)b * kChunkBytes : kWsW1);
    const uint32_t half = b < 8 ? kChunkHalf : kW1Half;
    for (int i = tid; i < rows * K / 2; i += kPrepThreads) {
        const int n = i / (K / 2), k = 2 * (i % (K / 2));
        const float *src = W + (int64_t)(row0 + n) * K + k;
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
    const float *b1, *W2, *b2;
    const unsigned char *ws;
    float *out;
};

// dynamic shared memory carve-up (bytes) for N nodes per graph
struct Smem {
    static constexpr uint32_t ring = 0;
    static constexpr uint32_t w1 = ring + kRing * kChunkBytes;
    static constexpr uint32_t bias = w1 + 2 * kW1Half;
    __host__ __device__ static uint32_t bias_bytes(int N) { return kGraphs * H * N * (N + 1) * 4; }
    __host__ __device__ static uint32_t stage(int N) { return bias + bias_bytes(N); }
    // K / V staging of the attention, or (during the relation MLP) one
    // prefetch slot of 16 features per compute thread plus its mask value
    __host__ __device__ static uint32_t stage_bytes(int N) {
        const uint32_t kv = kComputeWarps * 2 * N * DH * 4, mlp = kComputeThreads * (P + 1) * 4;
        return kv > mlp ? kv : mlp;
    }
    __host__ __device__ static uint32_t nodes(int N) { return stage(N) + stage_bytes(N); }
    __host__ __device__ static uint32_t nodes_bytes(int N) { return kGraphs * N * kNodeStride * 4; }
    // b1 [16], W2 transposed [16][4], b2 [4], gamma [96], beta [96], |gamma|max, |beta|max
    __host__ __device__ static uint32_t params(int N) { return nodes(N) + nodes_bytes(N); }
    static constexpr uint32_t params_bytes = (P + P * H + H + 2 * D + 2) * 4;
    __host__ __device__ static uint32_t rscale(int N) { return params(N) + params_bytes; }
    __host__ __device__ static uint32_t total(int N) { return rscale(N) + 128 * 4 + 16; }
};

struct Barriers {
    uint64_t wfull[kRing], wdone[kRing], afull[4], dfull[4], xfull, qkv, cfull, ofull, drain;
};

// Control thread: weight ring and every MMA issue, driven by mbarriers.
__device__ void control_loop(const Params &p, unsigned char *sm, Barriers &br, uint32_t tmem,
                             int n_my, int nblk, int32_t *err) {
    const int total = kChunks * n_my;
    // expected phase parity of each ring slot / MLP slot barrier, one bit per slot
    uint32_t ph_wfull = 0, ph_wdone = 0, ph_afull = 0;
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
            "l"(src0 + (size_t)(r % kChunks) * kChunkBytes), "r"(kChunkBytes), "r"(bar)
            : "memory");
    };
    int loaded = 0, issued = 0, refill = 0;
    for (; loaded < total && loaded < kRing; ++loaded) load(loaded);
    const uint32_t w1h = smem_u32(sm + Smem::w1), w1l = w1h + kW1Half;
    constexpr uint32_t idesc_w = idesc_f16(kNB, 128), idesc_m = idesc_f16(P, 128);
    bool bail = false;
    for (int t = 0; t < n_my && !bail; ++t) {
        int mlp_left = nblk;
        bool x_ok = false, c_ok = false;
        uint64_t idle_since = 0;
        uint32_t idle = 0;
        while (issued < kChunks * (t + 1) || mlp_left > 0) {
            bool progress = false;
            // relation-MLP blocks whose A operand is in TMEM
            for (int q = 0; q < 4 && mlp_left > 0; ++q) {
                if (mbar_test(&br.afull[q], (ph_afull >> q) & 1u)) {
                    ph_afull ^= 1u << q;
                    fence_after();
                    const uint32_t base = tmem + kColMlp + 32u * q;
                    const uint64_t bh = smem_desc(w1h, 128, 256), bl = smem_desc(w1l, 128, 256);
                    mma_ts(base + 16, base, bh, idesc_m, 0);
                    mma_ts(base + 16, base, bl, idesc_m, 1);
                    mma_ts(base + 16, base + 8, bh, idesc_m, 1);
                    mma_commit(&br.dfull[q]);
                    --mlp_left;
                    progress = true;
                }
            }
            // refill the ring slot of the oldest chunk whose MMAs are done
            if (refill < issued && loaded < total) {
                const int s = refill % kRing;
                if (mbar_test(&br.wdone[s], (ph_wdone >> s) & 1u)) {
                    ph_wdone ^= 1u << s;
                    load(loaded++);
                    ++refill;
                    progress = true;
                }
            }
            // the next weight chunk's MMAs
            if (issued < kChunks * (t + 1)) {
                const int c = issued % kChunks, s = issued % kRing;
                if (c < kQkvChunks && !x_ok) x_ok = mbar_test(&br.xfull, (uint32_t)t & 1u);
                if (c >= kQkvChunks && !c_ok) c_ok = mbar_test(&br.cfull, (uint32_t)t & 1u);
                const bool ready = c < kQkvChunks ? x_ok : c_ok;
                if (ready && mbar_test(&br.wfull[s], (ph_wfull >> s) & 1u)) {
                    ph_wfull ^= 1u << s;
                    fence_after();
                    const uint32_t bh = ring0 + (uint32_t)s * kChunkBytes, bl = bh + kChunkHalf;
                    const uint32_t d = tmem + (uint32_t)(c < kQkvChunks ? kNB * c : kNB * (c - 6));
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t ah = tmem + kColAhi + 8u * ks, al = tmem + kColAlo + 8u * ks;
                        const uint64_t dh = smem_desc(bh + 256u * ks, 128, (D / 8) * 128);
                        const uint64_t dl = smem_desc(bl + 256u * ks, 128, (D / 8) * 128);
                        mma_ts(d, ah, dh, idesc_w, ks > 0);
                        mma_ts(d, ah, dl, idesc_w, 1);
                        mma_ts(d, al, dh, idesc_w, 1);
                    }
                    mma_commit(&br.wdone[s]);
                    if (c == kQkvChunks - 1) mma_commit(&br.qkv);
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

__global__ void __launch_bounds__(kThreads, 1) dense_tc_kernel(const Params p) {
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ Barriers br;
    __shared__ uint32_t tmem_slot;
    __shared__ int32_t sw_s[5];
    __shared__ int32_t vmax_s[kGraphs];
    const int N = p.N, NN = N * N, NS = N + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp >> 2, lq = warp & 3;  // role quad; TMEM lane quarter (graph)
    const WsHeader *hd = reinterpret_cast<const WsHeader *>(p.ws);
    int32_t *err = const_cast<int32_t *>(&hd->err);
    float *prm = reinterpret_cast<float *>(sm + Smem::params(N));
    float *b1s = prm, *w2t = b1s + P, *b2s = w2t + P * H, *gam = b2s + H, *bet = gam + D;
    float *gb_max = bet + D;  // [0] max |gamma|, [1] max |beta|
    int32_t *rscale = reinterpret_cast<int32_t *>(sm + Smem::rscale(N));
    float *bias = reinterpret_cast<float *>(sm + Smem::bias);
    float *nodes_s = reinterpret_cast<float *>(sm + Smem::nodes(N));

    // ---- set-up: parameters, W1 image, barriers, TMEM
    for (int i = tid; i < P; i += kThreads) b1s[i] = p.b1[i];
    for (int i = tid; i < H * P; i += kThreads) w2t[(i % P) * H + i / P] = p.W2[i];  // [u][h]
    for (int i = tid; i < H; i += kThreads) b2s[i] = p.b2[i];
    for (int i = tid; i < D; i += kThreads) {
        gam[i] = p.ln_w[i];
        bet[i] = p.ln_b[i];
    }
    if (warp == 1) {
        float g = 0.f, bb = 0.f;
        for (int i = lane; i < D; i += 32) {
            g = fmaxf(g, fabsf(p.ln_w[i]));
            bb = fmaxf(bb, fabsf(p.ln_b[i]));
        }
        g = warp_max(g);
        bb = warp_max(bb);
        if (lane == 0) {
            gb_max[0] = g;
            gb_max[1] = bb;
        }
    }
    {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(p.ws + kWsW1);
        uint32_t *dst = reinterpret_cast<uint32_t *>(sm + Smem::w1);
        for (int i = tid; i < (int)(2 * kW1Half / 4); i += kThreads) dst[i] = src[i];
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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
        for (int q = 0; q < 4; ++q) {
            mbar_init(&br.afull[q], 128);
            mbar_init(&br.dfull[q], 1);
        }
        mbar_init(&br.xfull, 128);
        mbar_init(&br.qkv, 1);
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
    const int nblk = (kGraphs * NN + 127) / 128;  // relation-MLP blocks of 128 pairs per tile

    if (warp == kComputeWarps) {
        if (lane == 0) control_loop(p, sm, br, tmem, n_my, nblk, err);
        __syncwarp();
    } else {
        const uint32_t lane_q = (uint32_t)(32 * lq) << 16;  // this warp's TMEM lane quarter
        const float inv_sqrt_dh = 1.0f / sqrtf((float)DH);
        // relation-MLP blocks of this quad: quad 0 (after LayerNorm) the last k0,
        // quads 1-3 the rest round robin
        const int k0 = nblk / 6;
        const int mb_first = quad == 0 ? nblk - k0 : quad - 1;
        const int mb_step = quad == 0 ? 1 : 3;
        const int mb_end = quad == 0 ? nblk : nblk - k0;
        const uint32_t mslot = tmem + kColMlp + 32u * quad;
        uint32_t ph_dfull = 0;

        // node rows of tile `tile` into the staging buffer (quad 0)
        auto fetch_nodes = [&](int tile) {
            const int rows = kGraphs * N;
            for (int i = tid; i < rows * (D / 4); i += 128) {
                const int r = i / (D / 4), c = i % (D / 4), g = r / N;
                const int64_t b = (int64_t)tile * kGraphs + g;
                if (b < p.B)
                    cp_async16(smem_u32(nodes_s + r * kNodeStride + 4 * c),
                               p.nodes + (b * N + (r - g * N)) * (int64_t)D + 4 * c);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        if (quad == 0 && n_my > 0) fetch_nodes(blockIdx.x);
        // this thread's relation-MLP prefetch slot: 16 features and the mask value
        float *stage_base = reinterpret_cast<float *>(sm + Smem::stage(N));
        const float4 *pslot = reinterpret_cast<const float4 *>(stage_base + tid * P);
        const float *mslot_s = stage_base + kComputeThreads * P + tid;
        auto fetch_pair_block = [&](int tl, int blk) {
            const int pi = 128 * blk + 32 * lq + lane;
            const int64_t pg = (int64_t)tl * kGraphs * NN + pi;
            if (pi < kGraphs * NN && (int64_t)tl * kGraphs + pi / NN < p.B) {
#pragma unroll
                for (int c = 0; c < P / 4; ++c)
                    cp_async16(smem_u32(pslot + c), p.pair + pg * P + 4 * c);
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(mslot_s)),
                             "l"(p.mask + pg)
                             : "memory");
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };

        for (int it = 0; it < n_my; ++it) {
            const int tile = blockIdx.x + it * gridDim.x;
            const uint32_t par = (uint32_t)it & 1u;
            // ======== phase A: LayerNorm (quad 0) and the relation MLP (all)
            if (quad == 0) {
                asm volatile("cp.async.wait_all;" ::: "memory");
                named_sync(2, 128);
                const int g = lq, n = lane;
                const bool valid = (int64_t)tile * kGraphs + g < p.B && n < N;
                const float4 *xr =
                    reinterpret_cast<const float4 *>(nodes_s + (g * N + (valid ? n : 0)) * kNodeStride);
                float s1 = 0.f;
#pragma unroll 6
                for (int c = 0; c < D / 4; ++c) {
                    const float4 v = xr[c];
                    s1 += (v.x + v.y) + (v.z + v.w);
                }
                const float mean = s1 / (float)D;
                float v2 = 0.f, dmax = 0.f;
#pragma unroll 6
                for (int c = 0; c < D / 4; ++c) {
                    const float4 v = xr[c];
                    const float a0 = v.x - mean, a1 = v.y - mean, a2 = v.z - mean, a3 = v.w - mean;
                    v2 = fmaf(a0, a0, v2);
                    v2 = fmaf(a1, a1, v2);
                    v2 = fmaf(a2, a2, v2);
                    v2 = fmaf(a3, a3, v2);
                    dmax = fmaxf(dmax, fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(a2), fabsf(a3))));
                }
                const float rstd = 1.0f / sqrtf(v2 / (float)D + p.ln_eps);
                // an upper bound of |x_n| over the row picks its scale
                const int sr = valid ? scale_exp(dmax * rstd * gb_max[0] + gb_max[1]) : 0;
                const float sc = exp2i(sr);
                rscale[32 * g + n] = sr;
#pragma unroll 1
                for (int rd = 0; rd < D / 16; ++rd) {
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float4 v = xr[4 * rd + c];
                        const int k = 16 * rd + 4 * c;
                        float a[4] = {(v.x - mean) * rstd * gam[k] + bet[k],
                                      (v.y - mean) * rstd * gam[k + 1] + bet[k + 1],
                                      (v.z - mean) * rstd * gam[k + 2] + bet[k + 2],
                                      (v.w - mean) * rstd * gam[k + 3] + bet[k + 3]};
                        if (!valid) a[0] = a[1] = a[2] = a[3] = 0.f;
                        split2(a[0] * sc, a[1] * sc, hi[2 * c], lo[2 * c]);
                        split2(a[2] * sc, a[3] * sc, hi[2 * c + 1], lo[2 * c + 1]);
                    }
                    tmem_st8(tmem + lane_q + kColAhi + 8u * rd, hi);
                    tmem_st8(tmem + lane_q + kColAlo + 8u * rd, lo);
                }
                tmem_st_done();
                mbar_arrive(&br.xfull);
                if (tid < kGraphs) vmax_s[tid] = 0;
            }
            {
                // relation MLP: thread = pair (row 32 lq + lane of each 128-pair block);
                // the block's features and mask arrive in this thread's slot of
                // the staging region (idle until the attention) by cp.async,
                // the next block's while this one is computed
                if (mb_first < mb_end && it == 0) fetch_pair_block(tile, mb_first);
                for (int blk = mb_first; blk < mb_end; blk += mb_step) {
                    const int pi = 128 * blk + 32 * lq + lane;
                    const bool valid = pi < kGraphs * NN && (int64_t)tile * kGraphs + pi / NN < p.B;
                    asm volatile("cp.async.wait_all;" ::: "memory");
                    float pf[P];
#pragma unroll
                    for (int c = 0; c < P / 4; ++c) {
                        const float4 v = valid ? pslot[c] : make_float4(0.f, 0.f, 0.f, 0.f);
                        pf[4 * c] = v.x;
                        pf[4 * c + 1] = v.y;
                        pf[4 * c + 2] = v.z;
                        pf[4 * c + 3] = v.w;
                    }
                    const float mask_v = *mslot_s;
                    if (blk + mb_step < mb_end) fetch_pair_block(tile, blk + mb_step);
                    float m = 0.f;
#pragma unroll
                    for (int u = 0; u < P; ++u) m = fmaxf(m, fabsf(pf[u]));
                    const int sp = scale_exp(m);
                    {
                        const float sc = exp2i(sp);
                        uint32_t hi[8], lo[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            split2(pf[2 * c] * sc, pf[2 * c + 1] * sc, hi[c], lo[c]);
                        tmem_st8(mslot + lane_q, hi);
                        tmem_st8(mslot + lane_q + 8, lo);
                    }
                    tmem_st_done();
                    mbar_arrive(&br.afull[quad]);
                    mbar_wait(&br.dfull[quad], ph_dfull, err);
                    ph_dfull ^= 1u;
                    fence_after();
                    float hid[P];
                    tmem_ld16(mslot + lane_q + 16, hid);
                    const float unsc = exp2i(-sp) * exp2i(-sw_s[4]);
                    float r[H];
#pragma unroll
                    for (int h = 0; h < H; ++h) r[h] = b2s[h];
#pragma unroll
                    for (int u = 0; u < P; ++u) {
                        const float a = fmaf(hid[u], unsc, b1s[u]);
                        const float sl = __fdividef(a, 1.0f + __expf(-a));  // SiLU
                        const float4 w = *reinterpret_cast<const float4 *>(w2t + u * H);
                        r[0] = fmaf(w.x, sl, r[0]);
                        r[1] = fmaf(w.y, sl, r[1]);
                        r[2] = fmaf(w.z, sl, r[2]);
                        r[3] = fmaf(w.w, sl, r[3]);
                    }
                    if (valid) {
                        const int g = pi / NN, rem = pi - g * NN, n = rem / N, j = rem - n * N;
                        const bool masked = mask_v < 0.5f;
#pragma unroll
                        for (int h = 0; h < H; ++h)
                            bias[((g * H + h) * N + j) * NS + n] = masked ? -INFINITY : r[h];
                    }
                }
            }
            if (quad == 0 && it + 1 < n_my) fetch_nodes(tile + gridDim.x);  // LayerNorm is done
            named_sync(1, kComputeThreads);  // every pair's bias written
            mbar_wait(&br.qkv, par, err);
            fence_after();

            // ======== phase B: attention of head h = quad in graph g = lq
            const int g = lq, h = quad, n = lane;
            const int64_t b = (int64_t)tile * kGraphs + g;
            const bool rvalid = b < p.B && n < N;
            const int sr = rscale[32 * g + n];
            float ctx[DH];
            {
                float *sk = reinterpret_cast<float *>(sm + Smem::stage(N)) + warp * 2 * N * DH;
                float *sv = sk + N * DH;
                const float uq = exp2i(-sr) * exp2i(-sw_s[0]), uk = exp2i(-sr) * exp2i(-sw_s[1]),
                            uv = exp2i(-sr) * exp2i(-sw_s[2]);
                float q[DH];
                float vm = 0.f;
#pragma unroll
                for (int c0 = 0; c0 < DH; c0 += 8) {
                    float t8[8];
                    tmem_ld8(tmem + lane_q + (uint32_t)(h * DH + c0), q + c0);
#pragma unroll
                    for (int i = 0; i < 8; ++i) q[c0 + i] *= uq;
                    tmem_ld8(tmem + lane_q + (uint32_t)(D + h * DH + c0), t8);
                    if (rvalid) {
                        float4 *d4 = reinterpret_cast<float4 *>(sk + n * DH + c0);
                        d4[0] = make_float4(t8[0] * uk, t8[1] * uk, t8[2] * uk, t8[3] * uk);
                        d4[1] = make_float4(t8[4] * uk, t8[5] * uk, t8[6] * uk, t8[7] * uk);
                    }
                    tmem_ld8(tmem + lane_q + (uint32_t)(2 * D + h * DH + c0), t8);
                    if (rvalid) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            t8[i] *= uv;
                            vm = fmaxf(vm, fabsf(t8[i]));
                        }
                        float4 *d4 = reinterpret_cast<float4 *>(sv + n * DH + c0);
                        d4[0] = make_float4(t8[0], t8[1], t8[2], t8[3]);
                        d4[1] = make_float4(t8[4], t8[5], t8[6], t8[7]);
                    }
                }
                vm = warp_max(vm);
                if (lane == 0) atomicMax(&vmax_s[g], __float_as_int(vm));
                __syncwarp();
                // the score of (n, j) replaces its bias entry, which only this
                // lane reads: the two softmax passes keep no score registers
                float *brow = bias + (g * H + h) * N * NS + n;
                float m = -INFINITY;
                const int nj = rvalid ? N : 0;  // lanes past the graph's nodes touch nothing
#pragma unroll 4
                for (int j = 0; j < nj; ++j) {
                    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                    for (int c = 0; c < DH; c += 4) {
                        const float4 k4 = *reinterpret_cast<const float4 *>(sk + j * DH + c);
                        a0 = fmaf(q[c], k4.x, a0);
                        a1 = fmaf(q[c + 1], k4.y, a1);
                        a2 = fmaf(q[c + 2], k4.z, a2);
                        a3 = fmaf(q[c + 3], k4.w, a3);
                    }
                    const float s = ((a0 + a1) + (a2 + a3)) * inv_sqrt_dh + brow[j * NS];
                    brow[j * NS] = s;
                    m = fmaxf(m, s);
                }
#pragma unroll
                for (int c = 0; c < DH; ++c) ctx[c] = 0.f;
                float z = 0.f;
#pragma unroll 2
                for (int j = 0; j < nj; ++j) {
                    {
                        const float e = expf(brow[j * NS] - m);  // all -inf row: NaN, as the reference
                        z += e;
#pragma unroll
                        for (int c = 0; c < DH; c += 4) {
                            const float4 v4 = *reinterpret_cast<const float4 *>(sv + j * DH + c);
                            ctx[c] = fmaf(e, v4.x, ctx[c]);
                            ctx[c + 1] = fmaf(e, v4.y, ctx[c + 1]);
                            ctx[c + 2] = fmaf(e, v4.z, ctx[c + 2]);
                            ctx[c + 3] = fmaf(e, v4.w, ctx[c + 3]);
                        }
                    }
                }
                const float inv_z = 1.0f / z;
#pragma unroll
                for (int c = 0; c < DH; ++c) ctx[c] = rvalid ? ctx[c] * inv_z : 0.f;
            }
            named_sync(1, kComputeThreads);  // every graph's largest |V| known; staging free
            if (it + 1 < n_my && mb_first < mb_end) fetch_pair_block(tile + gridDim.x, mb_first);
            // the context (|ctx| <= max |V| of the graph) as the out-projection's A operand
            const int sc_g = scale_exp(__int_as_float(vmax_s[g]));
            {
                const float sc = exp2i(sc_g);
                uint32_t hi[DH / 2], lo[DH / 2];
#pragma unroll
                for (int c = 0; c < DH / 2; ++c)
                    split2(ctx[2 * c] * sc, ctx[2 * c + 1] * sc, hi[c], lo[c]);
#pragma unroll
                for (int c = 0; c < DH / 2; c += 4) {
                    tmem_st4(tmem + lane_q + kColAhi + (uint32_t)(h * DH / 2 + c), hi + c);
                    tmem_st4(tmem + lane_q + kColAlo + (uint32_t)(h * DH / 2 + c), lo + c);
                }
            }
            tmem_st_done();
            mbar_arrive(&br.cfull);

            // ======== phase C: out-projection columns [24h, 24h + 24) + residual
            mbar_wait(&br.ofull, par, err);
            fence_after();
            {
                const float fail = *reinterpret_cast<volatile int32_t *>(err) ? NAN : 0.f;
                const float uo = exp2i(-sc_g) * exp2i(-sw_s[3]);
                const float *x = p.nodes + (b * N + n) * (int64_t)D;
                float *o = p.out + (b * N + n) * (int64_t)D;
#pragma unroll
                for (int c0 = h * DH; c0 < (h + 1) * DH; c0 += 8) {
                    float v[8];
                    tmem_ld8(tmem + lane_q + (uint32_t)c0, v);
                    if (rvalid) {
                        const float4 x0 = __ldg(reinterpret_cast<const float4 *>(x + c0));
                        const float4 x1 = __ldg(reinterpret_cast<const float4 *>(x + c0 + 4));
                        reinterpret_cast<float4 *>(o + c0)[0] =
                            make_float4(fmaf(v[0], uo, x0.x) + fail, fmaf(v[1], uo, x0.y) + fail,
                                        fmaf(v[2], uo, x0.z) + fail, fmaf(v[3], uo, x0.w) + fail);
                        reinterpret_cast<float4 *>(o + c0)[1] =
                            make_float4(fmaf(v[4], uo, x1.x) + fail, fmaf(v[5], uo, x1.y) + fail,
                                        fmaf(v[6], uo, x1.z) + fail, fmaf(v[7], uo, x1.w) + fail);
                    }
                }
            }
            fence_before();
            named_sync(1, kComputeThreads);  // TMEM columns free for the next tile
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

// GAT_ERR_UNSUPPORTED when the shape is outside this path (the caller then
// runs the SIMT kernel).
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
    tc::dense_prep_kernel<<<9, tc::kPrepThreads, 0, s>>>(Wq, Wk, Wv, Wout, W1, ws);
    gat_status_t st = check_launch("gat_dense_masked_attention (weight prep)");
    if (st != GAT_OK) return st;
    const uint32_t smem = tc::Smem::total(N);
    static std::atomic<int> smem_set[kMaxDevices];
    cudaError_t e = allow_dynamic_smem(smem_set, tc::dense_tc_kernel, (int)tc::Smem::total(tc::kMaxN));
    if (e != cudaSuccess) return cuda_fail(e, "gat_dense_masked_attention: smem attribute");
    tc::Params p{B, N, nodes, pair, mask, ln_w, ln_b, ln_eps, b1, W2, b2, ws, out};
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
