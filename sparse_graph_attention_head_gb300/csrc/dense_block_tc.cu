// dense_block_tc.cu - the dense-masked attention block with its projections on
// the 5th-generation tensor cores (tcgen05, kind::tf32, accumulators in TMEM).
//
// The block page's module (Kimi-K2.6 l2_p4, reference model) spends three
// quarters of its arithmetic in four D x D projections (Q, K, V, out). Here they
// run as 128-row tcgen05 MMAs: a tile is 4 graphs, each padded to 32 rows, so
// graph g of the tile owns TMEM lanes 32g..32g+31 and is served by the four
// warps g, g+4, g+8, g+12 (the warps allowed to read that lane quarter). fp32
// accuracy comes from the 3xTF32 split: every operand x = hi + lo with
// hi = tf32(x) (round to nearest) and lo = x - hi, and
// A*B ~ hi_A hi_B + hi_A lo_B + lo_A hi_B (the dropped lo_A lo_B term and lo's
// own tf32 truncation are ~2^-20 relative).
//
// One CTA of 16 warps per SM, persistent over tiles. Warp w has lane quarter
// (graph) g = w % 4 and role group k = w / 4:
//   all    LayerNorm, warp w on the tile's 8-row group w -> hi/lo A operand
//          (shared memory, no-swizzle K-major 8-row x 16-byte core matrices)
//   k = 1  splits the weights into 48-column hi/lo B chunks (2-slot ring, the
//          next chunk's global loads in flight in registers) and, through its
//          first thread, issues each chunk's MMAs (commit -> one mbarrier per
//          ring slot)
//   k != 1 relation-MLP bias of the node pairs with the edge mask folded in
//          (-inf where masked), split evenly over groups 0, 2 and 3 (group 1
//          is streaming the Q|K|V weights meanwhile)
//   k      attention for head k: Q, K, V rows from TMEM, K and V staged in the
//          A region (idle once Q|K|V are in TMEM), scores + bias, softmax,
//          context kept in registers until every warp has read its staging,
//          then written as the hi/lo A operand of the out-projection
//   k = 1  out-projection chunks into the TMEM columns that held Q
//   k      residual add and store of output columns [kD/4, (k+1)D/4)
// Every mbarrier wait is bounded; a wait that gives up raises a device flag
// and the tile is written as NaN (never as silent garbage).
#include "common.cuh"

namespace gat {

namespace tc {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kGraphs = 4;      // graphs per tile (one 32-row TMEM lane quarter each)
constexpr int kRows = 128;      // MMA M
constexpr int kNB = 48;         // output columns per weight chunk (MMA N)
constexpr int kTmemCols = 512;  // Q|K|V need 3D columns
constexpr uint32_t kWaitTries = 1u << 24;

__device__ int g_tc_error;  // set when a bounded wait gives up

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of element (r, k) of a K-major tile whose rows have K elements
__device__ __forceinline__ uint32_t kmaj(int r, int k, int K) {
    return (uint32_t)((r >> 3) * (K >> 2) * 128 + (k >> 2) * 128 + (r & 7) * 16 + (k & 3) * 4);
}

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}

__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

__device__ __forceinline__ void split4(const float4 &v, float4 &hi, float4 &lo) {
    hi = make_float4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
    lo = make_float4(v.x - hi.x, v.y - hi.y, v.z - hi.z, v.w - hi.w);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         int accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// bounded wait for the completion of the phase with parity `parity`
__device__ __forceinline__ void mbar_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done = 0;
    for (uint32_t it = 0; it < kWaitTries && !done; ++it) {
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
    }
    if (!done) atomicExch(&g_tc_error, 1);
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 8 consecutive TMEM columns of this warp's 32 lanes
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

struct Params {
    int32_t B, N;
    const float *nodes, *pair, *mask, *ln_w, *ln_b;
    float ln_eps;
    const float *Wq, *Wk, *Wv, *W1, *b1, *W2, *b2, *Wout;
    float *out;
};

// Shared memory carve-up in bytes; tensor-core operands 1024-aligned.
template <int P, int H, int DH>
struct Smem {
    static constexpr int D = H * DH;
    static constexpr uint32_t kA = kRows * D * 4, kB = kNB * D * 4;
    static constexpr uint32_t al(uint32_t x) { return (x + 1023u) & ~1023u; }
    static constexpr uint32_t a_hi = 0, a_lo = al(a_hi + kA), b_hi0 = al(a_lo + kA),
                              b_lo0 = al(b_hi0 + kB), b_hi1 = al(b_lo0 + kB),
                              b_lo1 = al(b_hi1 + kB), mlp = al(b_lo1 + kB),
                              bias = mlp + (uint32_t)((P * P + P + H * P + H) * 4);
    // K/V staging of attention reuses [a_hi, a_lo + kA): 16 warps x 2 x N x DH floats
    __host__ __device__ static uint32_t stage_bytes(int N) { return kWarps * 2 * N * DH * 4; }
    __host__ __device__ static uint32_t total(int N) { return bias + kGraphs * H * N * N * 4; }
    __host__ __device__ static bool fits(int N) {
        return stage_bytes(N) <= a_lo + kA && total(N) <= 227u * 1024u - 64u;
    }
    __device__ static uint32_t b_hi(int s) { return s ? b_hi1 : b_hi0; }
    __device__ static uint32_t b_lo(int s) { return s ? b_lo1 : b_lo0; }
};

// Weight chunk `chunk` of [Wq; Wk; Wv] (chunk < 3D/kNB) or of Wout (after),
// split into the hi/lo B operand of ring slot s by the 128 threads of group 1
// (t = 0..127). Output column fastest across threads, so a warp's 16-byte
// shared stores land in distinct banks. Two steps, so the next chunk's global
// loads are in flight while the loader waits for its ring slot: fetch (global
// -> registers) and store (split -> shared memory).
template <int D>
struct ChunkRegs {
    static constexpr int kPer = kNB * (D / 4) / 128;  // float4 per loader thread
    static_assert(kNB * (D / 4) % 128 == 0, "chunk must split evenly over 128 threads");
    float4 w[kPer];
};

template <int P, int H, int DH>
__device__ __forceinline__ void fetch_chunk(const Params &p, int chunk, ChunkRegs<H * DH> &r,
                                            int t) {
    constexpr int D = H * DH, n_qkv = 3 * D / kNB;
#pragma unroll
    for (int i = 0; i < ChunkRegs<D>::kPer; ++i) {
        const int idx = t + 128 * i, o = idx % kNB, kg = idx / kNB;
        int row;
        const float *W;
        if (chunk < n_qkv) {
            const int rr = chunk * kNB + o;  // row of the stacked [Wq; Wk; Wv]
            W = rr < D ? p.Wq : (rr < 2 * D ? p.Wk : p.Wv);
            row = rr % D;
        } else {
            W = p.Wout;
            row = (chunk - n_qkv) * kNB + o;
        }
        r.w[i] = __ldg(reinterpret_cast<const float4 *>(W + (int64_t)row * D) + kg);
    }
}

template <int P, int H, int DH>
__device__ __forceinline__ void store_chunk(const ChunkRegs<H * DH> &r, unsigned char *sm, int s,
                                            int t) {
    using L = Smem<P, H, DH>;
    constexpr int D = L::D;
#pragma unroll
    for (int i = 0; i < ChunkRegs<D>::kPer; ++i) {
        const int idx = t + 128 * i, o = idx % kNB, kg = idx / kNB;
        float4 hi, lo;
        split4(r.w[i], hi, lo);
        const uint32_t off = kmaj(o, 4 * kg, D);
        *reinterpret_cast<float4 *>(sm + L::b_hi(s) + off) = hi;
        *reinterpret_cast<float4 *>(sm + L::b_lo(s) + off) = lo;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The 3xTF32 MMAs of one kNB-column chunk: D[:, col0:col0+kNB] = A B^T.
template <int D>
__device__ __forceinline__ void issue_chunk(uint32_t tmem, int col0, uint32_t a_hi, uint32_t a_lo,
                                            uint32_t b_hi, uint32_t b_lo) {
    constexpr uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) |
                               ((uint32_t)(kNB >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
    constexpr uint32_t lbo = 128, sbo = (uint32_t)(D / 4) * 128;
    const uint32_t d = tmem + (uint32_t)col0;
#pragma unroll
    for (int k0 = 0; k0 < D; k0 += 8) {
        const uint32_t ko = (uint32_t)(k0 / 4) * 128;
        const uint64_t ah = smem_desc(a_hi + ko, lbo, sbo), al = smem_desc(a_lo + ko, lbo, sbo);
        const uint64_t bh = smem_desc(b_hi + ko, lbo, sbo), bl = smem_desc(b_lo + ko, lbo, sbo);
        mma_tf32(d, ah, bh, idesc, k0 > 0);
        mma_tf32(d, ah, bl, idesc, 1);
        mma_tf32(d, al, bh, idesc, 1);
    }
}

// Relation-MLP bias of pairs (n, j), j in [j0, j1), for all heads, with the
// edge mask folded in (-inf where mask < 0.5); stored as
// bias_g[(h*N + j)*N + n] so a warp's lanes (n) write and read consecutive
// words. The next pair's features are loaded while the current one computes.
template <int P, int H>
__device__ __forceinline__ void mlp_bias(const float *prow, const float *mrow, int j0, int j1,
                                         const float *w1, const float *bb1, const float *w2,
                                         const float *bb2, float *bias_g, int N, int n) {
    // two pairs' features in flight ahead of the one being computed
    float4 nxt[P / 4], nxt2[P / 4];
#pragma unroll
    for (int c4 = 0; c4 < P / 4; ++c4) {
        nxt[c4] = j0 < j1 ? __ldg(reinterpret_cast<const float4 *>(prow + j0 * P) + c4)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        nxt2[c4] = j0 + 1 < j1 ? __ldg(reinterpret_cast<const float4 *>(prow + (j0 + 1) * P) + c4)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int j = j0; j < j1; ++j) {
        float pf[P];
#pragma unroll
        for (int c4 = 0; c4 < P / 4; ++c4) {
            pf[4 * c4] = nxt[c4].x;
            pf[4 * c4 + 1] = nxt[c4].y;
            pf[4 * c4 + 2] = nxt[c4].z;
            pf[4 * c4 + 3] = nxt[c4].w;
            nxt[c4] = nxt2[c4];
        }
        if (j + 2 < j1) {
#pragma unroll
            for (int c4 = 0; c4 < P / 4; ++c4)
                nxt2[c4] = __ldg(reinterpret_cast<const float4 *>(prow + (j + 2) * P) + c4);
        }
        float r[H];
#pragma unroll
        for (int h = 0; h < H; ++h) r[h] = bb2[h];
#pragma unroll
        for (int u = 0; u < P; ++u) {
            // W1 row u and W2 column u (stored transposed, w2t[u*H + h]) as
            // 16-byte shared-memory reads; even and odd products summed
            // apart, as before
            const float4 *w1r = reinterpret_cast<const float4 *>(w1 + u * P);
            float a0 = bb1[u], a1 = 0.f;
#pragma unroll
            for (int c4 = 0; c4 < P / 4; ++c4) {
                const float4 w = w1r[c4];
                a0 = fmaf(w.x, pf[4 * c4], a0);
                a1 = fmaf(w.y, pf[4 * c4 + 1], a1);
                a0 = fmaf(w.z, pf[4 * c4 + 2], a0);
                a1 = fmaf(w.w, pf[4 * c4 + 3], a1);
            }
            const float a = a0 + a1;
            const float hid = __fdividef(a, 1.0f + __expf(-a));  // SiLU
            const float4 w2c = *reinterpret_cast<const float4 *>(w2 + u * H);
            r[0] = fmaf(w2c.x, hid, r[0]);
            r[1] = fmaf(w2c.y, hid, r[1]);
            r[2] = fmaf(w2c.z, hid, r[2]);
            r[3] = fmaf(w2c.w, hid, r[3]);
        }
        const bool masked = __ldg(mrow + j) < 0.5f;
#pragma unroll
        for (int h = 0; h < H; ++h) bias_g[(h * N + j) * N + n] = masked ? -INFINITY : r[h];
    }
}

template <int P, int H, int DH>
__global__ void __launch_bounds__(kThreads, 1) dense_tc_kernel(const Params p) {
    using L = Smem<P, H, DH>;
    constexpr int D = L::D, n_qkv = 3 * D / kNB, n_out = D / kNB;
    static_assert(H == 4, "one attention head per role group");
    static_assert(P % 4 == 0, "16-byte reads of the relation-MLP weights");
    static_assert(3 * D % kNB == 0 && D % kNB == 0 && DH % 8 == 0, "chunking");
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ uint64_t bar[2];
    __shared__ uint32_t tmem_slot;
    const int N = p.N;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = warp & 3;   // graph of the tile / TMEM lane quarter
    const int grp = warp >> 2;  // role group, also the attention head
    const int tl = tid - 128;   // loader thread index (group 1)
    float *w1 = reinterpret_cast<float *>(sm + L::mlp), *bb1 = w1 + P * P, *w2 = bb1 + P,
          *bb2 = w2 + H * P;
    float *bias = reinterpret_cast<float *>(sm + L::bias);
    float *stage = reinterpret_cast<float *>(sm) + warp * 2 * N * DH;  // in the A region
    const uint32_t a_hi = smem_u32(sm + L::a_hi), a_lo = smem_u32(sm + L::a_lo);
    const float inv_sqrt_dh = 1.0f / sqrtf((float)DH);
    // relation-MLP pair ranges: groups 0, 2 and 3 split the pairs evenly;
    // group 1 streams the Q|K|V weight chunks meanwhile and takes none
    const int jb2 = 0, jb3 = N / 3, jb0 = (2 * N) / 3;
    const int j_lo = grp == 2 ? jb2 : grp == 3 ? jb3 : grp == 0 ? jb0 : N;
    const int j_hi = grp == 2 ? jb3 : grp == 3 ? jb0 : N;

    for (int i = tid; i < P * P; i += kThreads) w1[i] = p.W1[i];
    for (int i = tid; i < P; i += kThreads) bb1[i] = p.b1[i];
    for (int i = tid; i < H * P; i += kThreads) w2[(i % P) * H + i / P] = p.W2[i];  // [u][h]
    for (int i = tid; i < H; i += kThreads) bb2[i] = p.b2[i];
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[0])));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[1])));
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_slot;
    const uint32_t lane_q = (uint32_t)(32 * g) << 16;  // this warp's TMEM lane quarter
    uint32_t ncommit[2] = {0, 0};                       // commits issued per mbarrier

    const int n_tiles = (p.B + kGraphs - 1) / kGraphs;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int64_t b = (int64_t)tile * kGraphs + g;  // this warp's graph
        const int n = lane;                             // node row of this lane
        const bool rvalid = b < p.B && n < N;
        const int row = 32 * g + lane;                  // MMA row / TMEM lane
        const float *x = p.nodes + (b * N + n) * (int64_t)D;
        const float *prow = p.pair + ((b * N + n) * (int64_t)N) * P;
        float *bias_g = bias + g * H * N * N;

        // ---- LayerNorm -> A, all warps: warp w normalises the 8-row group w of the
        // tile (graph w/4, nodes 8(w%4)..+7); lane = (row r8 = lane%8, column
        // group cg = lane/8), column groups cg, cg+4, ... of 4 floats, so the
        // row loads are contiguous and the 16-byte A stores hit distinct banks.
        // Group 1 has weight chunk 0's loads in flight meanwhile.
        ChunkRegs<D> cr;
        if (grp == 1) fetch_chunk<P, H, DH>(p, 0, cr, tl);  // previous tile's MMAs are done
        {
            constexpr int NCG = D / 16;  // column groups per lane
            const int r8 = lane & 7, cg = lane >> 3;
            const int lg = warp >> 2, ln_node = 8 * (warp & 3) + r8;  // graph, node
            const int64_t lb = (int64_t)tile * kGraphs + lg;
            const bool lvalid = lb < p.B && ln_node < N;
            const int lrow = 32 * lg + ln_node;
            const float4 *xr = reinterpret_cast<const float4 *>(p.nodes + (lb * N + ln_node) * (int64_t)D);
            float4 xv[NCG];
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < NCG; ++i) {
                xv[i] = lvalid ? __ldg(xr + cg + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
                s += (xv[i].x + xv[i].y) + (xv[i].z + xv[i].w);
            }
            s += __shfl_xor_sync(kFull, s, 8);
            s += __shfl_xor_sync(kFull, s, 16);
            const float mean = s / (float)D;
            float v2 = 0.f;
#pragma unroll
            for (int i = 0; i < NCG; ++i) {
                const float a0 = xv[i].x - mean, a1 = xv[i].y - mean, a2 = xv[i].z - mean,
                            a3 = xv[i].w - mean;
                v2 = fmaf(a0, a0, v2);
                v2 = fmaf(a1, a1, v2);
                v2 = fmaf(a2, a2, v2);
                v2 = fmaf(a3, a3, v2);
            }
            v2 += __shfl_xor_sync(kFull, v2, 8);
            v2 += __shfl_xor_sync(kFull, v2, 16);
            const float rstd = 1.0f / sqrtf(v2 / (float)D + p.ln_eps);
#pragma unroll
            for (int i = 0; i < NCG; ++i) {
                const int k4 = cg + 4 * i;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                if (lvalid) {
                    const float4 gw = __ldg(reinterpret_cast<const float4 *>(p.ln_w) + k4);
                    const float4 gb = __ldg(reinterpret_cast<const float4 *>(p.ln_b) + k4);
                    a = make_float4((xv[i].x - mean) * rstd * gw.x + gb.x,
                                    (xv[i].y - mean) * rstd * gw.y + gb.y,
                                    (xv[i].z - mean) * rstd * gw.z + gb.z,
                                    (xv[i].w - mean) * rstd * gw.w + gb.w);
                }
                float4 hi, lo;
                split4(a, hi, lo);
                const uint32_t off = kmaj(lrow, 4 * k4, D);
                *reinterpret_cast<float4 *>(sm + L::a_hi + off) = hi;
                *reinterpret_cast<float4 *>(sm + L::a_lo + off) = lo;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        if (grp == 1) {
            store_chunk<P, H, DH>(cr, sm, 0, tl);
            fetch_chunk<P, H, DH>(p, 1, cr, tl);
        }
        __syncthreads();  // A operand and chunk 0 in shared memory

        // ---- Q|K|V (group 1 streams chunks and issues) and the relation MLP
        if (grp == 1) {
            for (int c = 0; c < n_qkv; ++c) {
                const int s = c & 1;
                if (c > 0) {
                    if (c >= 2) mbar_wait(&bar[s], (ncommit[s] - 1) & 1);  // chunk c-2 done
                    store_chunk<P, H, DH>(cr, sm, s, tl);
                    if (c + 1 < n_qkv) fetch_chunk<P, H, DH>(p, c + 1, cr, tl);
                }
                named_sync(1, 128);
                if (tid == 128) {
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    issue_chunk<D>(tmem, c * kNB, a_hi, a_lo, smem_u32(sm + L::b_hi(s)),
                                   smem_u32(sm + L::b_lo(s)));
                    mma_commit(&bar[s]);
                }
                ++ncommit[s];
            }
        } else {
            ncommit[0] += (n_qkv + 1) / 2;
            ncommit[1] += n_qkv / 2;
        }
        if (rvalid)
            mlp_bias<P, H>(prow, p.mask + (b * N + n) * (int64_t)N, j_lo, j_hi, w1, bb1, w2, bb2,
                           bias_g, N, n);
        __syncthreads();  // bias complete
        {
            const int s = (n_qkv - 1) & 1;  // the last commit covers every earlier MMA
            mbar_wait(&bar[s], (ncommit[s] - 1) & 1);
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

        // ---- attention, head h = grp: K, V staged in the (now idle) A region
        const int h = grp;
        float ctx[DH];
        {
            float *sk = stage, *sv = stage + N * DH;
            float q[DH], kv[8];
#pragma unroll
            for (int c0 = 0; c0 < DH; c0 += 8) {
                tmem_ld8(tmem + lane_q + (uint32_t)(h * DH + c0), q + c0);
                tmem_ld8(tmem + lane_q + (uint32_t)(D + h * DH + c0), kv);
                if (rvalid) {
                    float4 *d4 = reinterpret_cast<float4 *>(sk + n * DH + c0);
                    d4[0] = make_float4(kv[0], kv[1], kv[2], kv[3]);
                    d4[1] = make_float4(kv[4], kv[5], kv[6], kv[7]);
                }
                tmem_ld8(tmem + lane_q + (uint32_t)(2 * D + h * DH + c0), kv);
                if (rvalid) {
                    float4 *d4 = reinterpret_cast<float4 *>(sv + n * DH + c0);
                    d4[0] = make_float4(kv[0], kv[1], kv[2], kv[3]);
                    d4[1] = make_float4(kv[4], kv[5], kv[6], kv[7]);
                }
            }
            __syncwarp();
            float sc[32];
            float m = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                float s = -INFINITY;
                if (j < N && rvalid) {
                    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                    for (int c = 0; c < DH; c += 4) {
                        const float4 k4 = *reinterpret_cast<const float4 *>(sk + j * DH + c);
                        a0 = fmaf(q[c], k4.x, a0);
                        a1 = fmaf(q[c + 1], k4.y, a1);
                        a2 = fmaf(q[c + 2], k4.z, a2);
                        a3 = fmaf(q[c + 3], k4.w, a3);
                    }
                    s = ((a0 + a1) + (a2 + a3)) * inv_sqrt_dh + bias_g[(h * N + j) * N + n];
                }
                sc[j] = s;
                m = fmaxf(m, s);
            }
            float z = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float e = (j < N) ? expf(sc[j] - m) : 0.f;  // all -inf row: NaN
                sc[j] = e;
                z += e;
            }
            const float inv_z = 1.0f / z;
#pragma unroll
            for (int c = 0; c < DH; ++c) ctx[c] = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j < N) {
                    const float a = sc[j] * inv_z;
#pragma unroll
                    for (int c = 0; c < DH; c += 4) {
                        const float4 v4 = *reinterpret_cast<const float4 *>(sv + j * DH + c);
                        ctx[c] = fmaf(a, v4.x, ctx[c]);
                        ctx[c + 1] = fmaf(a, v4.y, ctx[c + 1]);
                        ctx[c + 2] = fmaf(a, v4.z, ctx[c + 2]);
                        ctx[c + 3] = fmaf(a, v4.w, ctx[c + 3]);
                    }
                }
            }
        }
        if (grp == 1) fetch_chunk<P, H, DH>(p, n_qkv, cr, tl);  // out-projection chunk 0
        __syncthreads();  // every warp is done with its staging: A region free again
#pragma unroll
        for (int c = 0; c < DH; c += 4) {
            const float4 v = rvalid ? make_float4(ctx[c], ctx[c + 1], ctx[c + 2], ctx[c + 3])
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            float4 hi, lo;
            split4(v, hi, lo);
            const uint32_t off = kmaj(row, h * DH + c, D);
            *reinterpret_cast<float4 *>(sm + L::a_hi + off) = hi;
            *reinterpret_cast<float4 *>(sm + L::a_lo + off) = lo;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();

        // ---- out = ctx Wout^T into TMEM columns [0, D) (Q is no longer read)
        if (grp == 1) {
            for (int c = 0; c < n_out; ++c) {
                const int s = c & 1;
                if (c >= 2) mbar_wait(&bar[s], (ncommit[s] - 1) & 1);
                store_chunk<P, H, DH>(cr, sm, s, tl);
                if (c + 1 < n_out) fetch_chunk<P, H, DH>(p, n_qkv + c + 1, cr, tl);
                named_sync(1, 128);
                if (tid == 128) {
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    issue_chunk<D>(tmem, c * kNB, a_hi, a_lo, smem_u32(sm + L::b_hi(s)),
                                   smem_u32(sm + L::b_lo(s)));
                    mma_commit(&bar[s]);
                }
                ++ncommit[s];
            }
        } else {
            ncommit[0] += (n_out + 1) / 2;
            ncommit[1] += n_out / 2;
        }
        __syncthreads();
        {
            const int s = (n_out - 1) & 1;
            mbar_wait(&bar[s], (ncommit[s] - 1) & 1);
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

        // ---- residual add and store of columns [grp*D/4, (grp+1)*D/4); a tile whose
        // MMA wait gave up is written as NaN, never as silent garbage
        {
            const float fail = *reinterpret_cast<volatile int *>(&g_tc_error) ? NAN : 0.f;
            float *o = p.out + (b * N + n) * (int64_t)D;
#pragma unroll
            for (int c0 = grp * (D / 4); c0 < (grp + 1) * (D / 4); c0 += 8) {
                float v[8];
                tmem_ld8(tmem + lane_q + (uint32_t)c0, v);
                if (rvalid) {
                    const float4 x0 = __ldg(reinterpret_cast<const float4 *>(x + c0));
                    const float4 x1 = __ldg(reinterpret_cast<const float4 *>(x + c0 + 4));
                    reinterpret_cast<float4 *>(o + c0)[0] =
                        make_float4(x0.x + v[0] + fail, x0.y + v[1] + fail, x0.z + v[2] + fail,
                                    x0.w + v[3] + fail);
                    reinterpret_cast<float4 *>(o + c0)[1] =
                        make_float4(x1.x + v[4] + fail, x1.y + v[5] + fail, x1.z + v[6] + fail,
                                    x1.w + v[7] + fail);
                }
            }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
    }
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
}

}  // namespace tc

// Host side: GAT_ERR_UNSUPPORTED when the shape is outside this path (the
// caller then runs the SIMT kernel). This build instantiates P=16, H=4,
// head_dim=24 (D=96), the block page's module shape, for up to 28 nodes.
gat_status_t dense_block_tc(int32_t B, int32_t N, int32_t D, int32_t H, int32_t P,
                            const float *nodes, const float *pair, const float *mask,
                            const float *ln_w, const float *ln_b, float ln_eps, const float *Wq,
                            const float *Wk, const float *Wv, const float *W1, const float *b1,
                            const float *W2, const float *b2, const float *Wout, float *out,
                            cudaStream_t s) {
    constexpr int kP = 16, kH = 4, kDH = 24;
    using L = tc::Smem<kP, kH, kDH>;
    if (P != kP || H != kH || D != kH * kDH || N < 1 || N > 32 || !L::fits(N))
        return GAT_ERR_UNSUPPORTED;
    const uint32_t smem = L::total(N);
    auto kern = tc::dense_tc_kernel<kP, kH, kDH>;
    static uint32_t configured = 0;
    if (smem > configured) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_fail(e, "gat_dense_masked_attention: smem attribute");
        configured = smem;
    }
    int zero = 0;
    cudaError_t e = cudaMemcpyToSymbolAsync(tc::g_tc_error, &zero, sizeof(int), 0,
                                            cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "gat_dense_masked_attention: error flag");
    tc::Params p{B, N, nodes, pair, mask, ln_w, ln_b, ln_eps, Wq, Wk, Wv, W1, b1, W2, b2, Wout, out};
    const int64_t tiles = (B + tc::kGraphs - 1) / tc::kGraphs;
    int64_t blocks = sm_count();
    if (blocks > tiles) blocks = tiles;
    kern<<<(unsigned)blocks, tc::kThreads, smem, s>>>(p);
    return check_launch("gat_dense_masked_attention (tcgen05)");
}

}  // namespace gat
