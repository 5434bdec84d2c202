// fused_fp8.cu - the fused layer over fp8 (E4M3) k and v tables, and the
// quantiser that makes them.
//
// In the fused layer (POPCORNBENCH FW-GLM-5-1 l1_p6 / l1_p10 / l1_p18,
// reference models: score, softmax, aggregation) the per-edge gathers of the
// k and v rows are nearly all of the bytes. Stored as E4M3 with one fp32
// scale per (node, head), a 1 KB bf16 row becomes 512 B + 4H B, so a layer
// moves about 1.1 KB per edge instead of 2 KB. q and out stay in the layer's
// dtype; every sum is fp32.
//
//   gat_quantize_fp8: scale[n,h] = max_d |x[n,h,d]| / 448 (1 for an all-zero
//     head), code = E4M3(x / scale), nearest-even, saturating (448 is the
//     largest finite E4M3 magnitude); one warp per node row with 16-byte
//     loads when a head is a power-of-two number of vectors, else one warp
//     per (node, head).
//   gat_fused_layer_fp8: gat_fused_layer's lane layout with 16-byte vectors
//     of 16 fp8 elements: lane l of a warp holds vectors l, l+32 (V per lane)
//     of the row's H*Dh codes; a head is Dh/16 adjacent lanes. Per edge:
//     s = scale * ks[src,h] * <q, decode(k8[src])>, online softmax in log2
//     units, acc += p * vs[src,h] * decode(v8[src]). Heavy rows of a plan are
//     cut into chunks whose states merge exactly as in gat_fused_layer.
//     Wider rows run as groups of heads of 512 or 1024 codes, one launch per
//     group; other shapes take a scalar kernel (one warp per row, heads in
//     turn).
#include <climits>
#include <cuda_fp8.h>

#include "row_engine.cuh"

namespace gat {

constexpr int kFp8Threads = 128;
constexpr float kLog2e8 = 1.4426950408889634f;

struct Fp8Params {
    const int32_t *row_ptr, *col_idx;
    const void *q;  // [n_rows,H,Dh], T
    const uint8_t *k8, *v8;  // [n_src,H,Dh] E4M3 codes
    const float *ks, *vs;    // [n_src,H]
    void *out;               // [n_rows,H,Dh], T
    int64_t n_rows;
    int32_t H, Dh;
    int32_t Hs;    // heads per row of q, out, the code tables and the scales (H, or
                   // more for a head group whose slices start at head 0 of each row)
    float qscale;  // scale * log2(e)
    int32_t heavy_threshold;
    int64_t n_chunks;
    const int4 *chunk_desc;
    const int32_t *chunk_start;
    int32_t *counters;
    float *partials;  // [n_chunks][slot_floats]: acc [H*Dh], m [H], l [H]
    int64_t slot_floats;
};

// 16 E4M3 codes -> 8 float pairs (elements 2i, 2i + 1); exact: every E4M3 value is a half
__device__ __forceinline__ void decode16x2(const uint4 &u, float2 *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const __nv_fp8x2_storage_t pr = (__nv_fp8x2_storage_t)(w[i] >> (16 * j));
            f[2 * i + j] = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3)));
        }
}

// packed fp32 FMA on a pair, (a.x b.x + c.x, a.y b.y + c.y), each rounded once
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(r)
        : "l"(*reinterpret_cast<uint64_t *>(&a)), "l"(*reinterpret_cast<uint64_t *>(&b)),
          "l"(*reinterpret_cast<uint64_t *>(&c)));
    return *reinterpret_cast<float2 *>(&r);
}

// 16 consecutive elements of a T row, as floats
template <typename T>
__device__ __forceinline__ void load16(const T *p, float *f) {
    constexpr int NV = 16 / Vec<T>::N;  // 16-byte vectors
#pragma unroll
    for (int i = 0; i < NV; ++i)
        Vec<T>::unpack(ld_stream16(reinterpret_cast<const char *>(p) + 16 * i), f + i * Vec<T>::N);
}

template <typename T>
__device__ __forceinline__ void store16(T *p, const float *f) {
    constexpr int NV = 16 / Vec<T>::N;
#pragma unroll
    for (int i = 0; i < NV; ++i)
        st_stream16(reinterpret_cast<char *>(p) + 16 * i, Vec<T>::pack(f + i * Vec<T>::N));
}

template <typename T, int V, int U>
struct Fp8Row {
    float2 qf[V][8], acc[V][8];  // element pairs (packed fp32 arithmetic)
    float m[V], l[V];
    int lane, G, vi[V], head[V];

    __device__ __forceinline__ Fp8Row(int Dh) {
        lane = threadIdx.x & 31;
        G = Dh / 16;
#pragma unroll
        for (int s = 0; s < V; ++s) {
            vi[s] = s * 32 + lane;
            head[s] = vi[s] / G;
        }
    }

    __device__ __forceinline__ void begin(const Fp8Params &p, int64_t row) {
        const T *qrow = static_cast<const T *>(p.q) + row * (int64_t)p.Hs * p.Dh;
#pragma unroll
        for (int s = 0; s < V; ++s) {
            float qv[16];
            load16(qrow + vi[s] * 16, qv);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                qf[s][t] = make_float2(qv[2 * t] * p.qscale, qv[2 * t + 1] * p.qscale);
                acc[s][t] = make_float2(0.f, 0.f);
            }
            m[s] = -INFINITY;
            l[s] = 0.f;
        }
    }

    __device__ __forceinline__ void run(const Fp8Params &p, int e0, int e1) {
        const int64_t HD = (int64_t)p.Hs * p.Dh;
        for (int base = e0; base < e1; base += 32) {
            const int n = min(32, e1 - base);
            const int my_ci = lane < n ? __ldg(p.col_idx + base + lane) : 0;
            for (int j0 = 0; j0 < n; j0 += U) {
                uint4 kr[U][V], vr[U][V];
                float kss[U][V], vss[U][V];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t src = __shfl_sync(kFull, my_ci, (j0 + u) & 31);
#pragma unroll
                    for (int s = 0; s < V; ++s) {
                        if (j0 + u < n) {
                            kr[u][s] = ld_stream16(p.k8 + src * HD + vi[s] * 16);
                            vr[u][s] = ld_stream16(p.v8 + src * HD + vi[s] * 16);
                            kss[u][s] = __ldg(p.ks + src * p.Hs + head[s]);
                            vss[u][s] = __ldg(p.vs + src * p.Hs + head[s]);
                        } else {
                            kr[u][s] = vr[u][s] = make_uint4(0, 0, 0, 0);
                            kss[u][s] = vss[u][s] = 0.f;
                        }
                    }
                }
                float sc[U][V];
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int s = 0; s < V; ++s) {
                        float2 kf[8];
                        decode16x2(kr[u][s], kf);
                        float2 d = make_float2(0.f, 0.f);
#pragma unroll
                        for (int t = 0; t < 8; ++t) d = fma2(qf[s][t], kf[t], d);
                        sc[u][s] = d.x + d.y;
                    }
                for (int o = 1; o < G; o <<= 1) {
#pragma unroll
                    for (int u = 0; u < U; ++u)
#pragma unroll
                        for (int s = 0; s < V; ++s) sc[u][s] += __shfl_xor_sync(kFull, sc[u][s], o);
                }
#pragma unroll
                for (int s = 0; s < V; ++s) {
                    float mx = m[s];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        sc[u][s] *= kss[u][s];
                        if (j0 + u < n) mx = fmaxf(mx, sc[u][s]);
                    }
                    if (mx == -INFINITY) continue;
                    const float c = fast_exp2(m[s] - mx);
                    l[s] *= c;
                    const float2 c2 = make_float2(c, c), z2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int t = 0; t < 8; ++t) acc[s][t] = fma2(acc[s][t], c2, z2);
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const float pe = j0 + u < n ? fast_exp2(sc[u][s] - mx) : 0.f;
                        l[s] += pe;
                        const float w = pe * vss[u][s];
                        const float2 w2 = make_float2(w, w);
                        float2 vf[8];
                        decode16x2(vr[u][s], vf);
#pragma unroll
                        for (int t = 0; t < 8; ++t) acc[s][t] = fma2(w2, vf[t], acc[s][t]);
                    }
                    m[s] = mx;
                }
            }
        }
    }

    __device__ __forceinline__ void store_out(const Fp8Params &p, int64_t row) {
        T *orow = static_cast<T *>(p.out) + row * (int64_t)p.Hs * p.Dh;
#pragma unroll
        for (int s = 0; s < V; ++s) {
            const float inv = l[s] > 0.f ? 1.f / l[s] : 0.f;
            float o[16];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                o[2 * t] = acc[s][t].x * inv;
                o[2 * t + 1] = acc[s][t].y * inv;
            }
            store16(orow + vi[s] * 16, o);
        }
    }

    // a chunk of a heavy row: publish (acc, m, l); the last chunk to finish
    // merges the row's chunk states in chunk order
    __device__ __forceinline__ void chunk_epilogue(const Fp8Params &p, int64_t row, int hr,
                                                   int64_t chunk) {
        const int HD = p.H * p.Dh;
        float *slot = p.partials + chunk * p.slot_floats;
#pragma unroll
        for (int s = 0; s < V; ++s) {
#pragma unroll
            for (int t = 0; t < 8; t += 2)
                __stcg(reinterpret_cast<float4 *>(slot + vi[s] * 16 + 2 * t),
                       make_float4(acc[s][t].x, acc[s][t].y, acc[s][t + 1].x, acc[s][t + 1].y));
            if (vi[s] % G == 0) {
                __stcg(slot + HD + head[s], m[s]);
                __stcg(slot + HD + p.H + head[s], l[s]);
            }
        }
        __threadfence();
        __syncwarp();
        int old = 0;
        if (lane == 0) old = atomicAdd(p.counters + hr, 1);
        old = __shfl_sync(kFull, old, 0);
        const int c0 = __ldg(p.chunk_start + hr), c1 = __ldg(p.chunk_start + hr + 1);
        if (old != c1 - c0 - 1) return;
        __threadfence();
#pragma unroll
        for (int s = 0; s < V; ++s) {
            m[s] = -INFINITY;
            l[s] = 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t) acc[s][t] = make_float2(0.f, 0.f);
        }
        for (int c = c0; c < c1; ++c) {
            const float *sl = p.partials + (int64_t)c * p.slot_floats;
#pragma unroll
            for (int s = 0; s < V; ++s) {
                const float mc = __ldcg(sl + HD + head[s]);
                const float lc = __ldcg(sl + HD + p.H + head[s]);
                const float mx = fmaxf(m[s], mc);
                if (mx == -INFINITY) continue;
                const float a1 = fast_exp2(m[s] - mx), a2 = fast_exp2(mc - mx);
                l[s] = l[s] * a1 + lc * a2;
#pragma unroll
                for (int t = 0; t < 8; t += 2) {
                    const float4 f = ld_cg_f4(sl + vi[s] * 16 + 2 * t);
                    acc[s][t].x = acc[s][t].x * a1 + f.x * a2;
                    acc[s][t].y = acc[s][t].y * a1 + f.y * a2;
                    acc[s][t + 1].x = acc[s][t + 1].x * a1 + f.z * a2;
                    acc[s][t + 1].y = acc[s][t + 1].y * a1 + f.w * a2;
                }
                m[s] = mx;
            }
        }
        store_out(p, row);
        if (lane == 0) p.counters[hr] = 0;  // ready for the next call
    }
};

// persistent: warp w takes items w, w + W, ... (chunks of heavy rows first,
// then every row; heavy rows skipped)
template <typename T, int V, int U>
__global__ void __launch_bounds__(kFp8Threads, V == 1 ? 5 : 3)
fused_fp8_kernel(const Fp8Params p) {
    Fp8Row<T, V, U> st(p.Dh);
    const int64_t wpb = blockDim.x >> 5;
    const int64_t n_warps = (int64_t)gridDim.x * wpb;
    const int64_t n_items = p.n_chunks + p.n_rows;
    for (int64_t item = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5); item < n_items;
         item += n_warps) {
        if (item < p.n_chunks) {
            const int4 d = __ldg(p.chunk_desc + item);
            st.begin(p, d.x);
            st.run(p, d.y, d.z);
            st.chunk_epilogue(p, d.x, d.w, item);
        } else {
            const int64_t row = item - p.n_chunks;
            const int e0 = __ldg(p.row_ptr + row), e1 = __ldg(p.row_ptr + row + 1);
            if (e1 - e0 > p.heavy_threshold) continue;
            st.begin(p, row);
            st.run(p, e0, e1);
            st.store_out(p, row);
        }
    }
}

// any shape: one warp per row, heads in turn, lanes over Dh (up to 8 each)
template <typename T>
__global__ void __launch_bounds__(kFp8Threads)
fused_fp8_generic_kernel(const Fp8Params p) {
    constexpr int MAXT = 8;
    const int lane = threadIdx.x & 31;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t n_warps = (int64_t)gridDim.x * wpb;
    const T *q = static_cast<const T *>(p.q);
    T *out = static_cast<T *>(p.out);
    const int64_t HD = (int64_t)p.H * p.Dh;
    for (int64_t row = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5); row < p.n_rows;
         row += n_warps) {
        const int e0 = __ldg(p.row_ptr + row), e1 = __ldg(p.row_ptr + row + 1);
        for (int h = 0; h < p.H; ++h) {
            const int64_t qo = row * HD + (int64_t)h * p.Dh;
            float qf[MAXT], acc[MAXT];
#pragma unroll
            for (int t = 0; t < MAXT; ++t) {
                const int d = lane + 32 * t;
                qf[t] = d < p.Dh ? load_elem(q, qo + d) * p.qscale : 0.f;
                acc[t] = 0.f;
            }
            float m = -INFINITY, l = 0.f;
            for (int e = e0; e < e1; ++e) {
                const int64_t src = __ldg(p.col_idx + e);
                const int64_t ko = src * HD + (int64_t)h * p.Dh;
                float d0 = 0.f;
#pragma unroll
                for (int t = 0; t < MAXT; ++t) {
                    const int d = lane + 32 * t;
                    if (d < p.Dh)
                        d0 = fmaf(qf[t],
                                  __half2float(__half(__nv_cvt_fp8_to_halfraw(p.k8[ko + d], __NV_E4M3))),
                                  d0);
                }
                const float sc = warp_sum(d0) * __ldg(p.ks + src * p.H + h);
                const float mx = fmaxf(m, sc);
                const float c = fast_exp2(m - mx), pe = fast_exp2(sc - mx);
                l = l * c + pe;
                const float w = pe * __ldg(p.vs + src * p.H + h);
#pragma unroll
                for (int t = 0; t < MAXT; ++t) {
                    const int d = lane + 32 * t;
                    const float vv =
                        d < p.Dh ? __half2float(__half(__nv_cvt_fp8_to_halfraw(p.v8[ko + d], __NV_E4M3)))
                                 : 0.f;
                    acc[t] = fmaf(w, vv, acc[t] * c);
                }
                m = mx;
            }
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int t = 0; t < MAXT; ++t) {
                const int d = lane + 32 * t;
                if (d < p.Dh) store_elem(out, qo + d, acc[t] * inv);
            }
        }
    }
}

// quantiser: one warp per (node, head), lanes over Dh
template <typename T>
__global__ void __launch_bounds__(256)
quantize_fp8_kernel(const T *__restrict__ x, int64_t n, int32_t H, int32_t Dh,
                    uint8_t *__restrict__ codes, float *__restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t pairs = n * H;
    for (int64_t ph = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); ph < pairs;
         ph += n_warps) {
        const int64_t o = ph * Dh;
        float amax = 0.f;
        for (int d = lane; d < Dh; d += 32) amax = fmaxf(amax, fabsf(load_elem(x, o + d)));
        amax = warp_max(amax);
        const float sc = amax > 0.f ? amax / 448.f : 1.f;  // IEEE division
        if (lane == 0) scales[ph] = sc;
        for (int d = lane; d < Dh; d += 32)
            codes[o + d] = __nv_cvt_float_to_fp8(load_elem(x, o + d) / sc, __NV_SATFINITE, __NV_E4M3);
    }
}

// quantiser, vector form: one warp per node row; lane l takes 16-byte vectors
// l, l+32, ... of the row; a head is G = Dh/VE adjacent lanes (G a power of
// two), so its maximum is a G-lane shuffle; each vector's VE codes leave as
// one VE-byte store.
template <typename T>
__global__ void __launch_bounds__(256)
quantize_fp8_vec_kernel(const T *__restrict__ x, int64_t n, int32_t H, int32_t Dh,
                        uint8_t *__restrict__ codes, float *__restrict__ scales) {
    constexpr int VE = Vec<T>::N;
    const int lane = threadIdx.x & 31;
    const int G = Dh / VE;
    const int nvec = H * G;  // vectors per row, a multiple of G
    const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < n;
         row += n_warps) {
        const char *xr = reinterpret_cast<const char *>(x + row * (int64_t)H * Dh);
        for (int j0 = 0; j0 < nvec; j0 += 32) {  // warp-uniform
            const int j = j0 + lane;
            float f[VE];
            if (j < nvec) {
                Vec<T>::unpack(ld_stream16(xr + (int64_t)j * 16), f);
            } else {
#pragma unroll
                for (int t = 0; t < VE; ++t) f[t] = 0.f;
            }
            float amax = 0.f;
#pragma unroll
            for (int t = 0; t < VE; ++t) amax = fmaxf(amax, fabsf(f[t]));
            for (int o = 1; o < G; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
            if (j >= nvec) continue;
            const float sc = amax > 0.f ? amax / 448.f : 1.f;  // IEEE division
            if (j % G == 0) scales[row * H + j / G] = sc;
            uint32_t w[VE / 4];
#pragma unroll
            for (int t = 0; t < VE; t += 4) {
                uint32_t b = 0;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    b |= (uint32_t)__nv_cvt_float_to_fp8(f[t + u] / sc, __NV_SATFINITE, __NV_E4M3)
                         << (8 * u);
                w[t / 4] = b;
            }
            uint8_t *cr = codes + row * (int64_t)H * Dh + (int64_t)j * VE;
            if (VE == 8)
                *reinterpret_cast<uint2 *>(cr) = make_uint2(w[0], w[VE / 4 - 1]);
            else
                *reinterpret_cast<uint32_t *>(cr) = w[0];
        }
    }
}

template <typename T, int V>
static gat_status_t launch_fp8_fast(const Fp8Params &p, cudaStream_t s) {
    constexpr int U = V == 1 ? 4 : 2;
    auto kern = fused_fp8_kernel<T, V, U>;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFp8Threads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t wpb = kFp8Threads / 32;
    int64_t blocks = (p.n_chunks + p.n_rows + wpb - 1) / wpb;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    if (blocks > cap) blocks = cap;
    kern<<<(unsigned)blocks, kFp8Threads, 0, s>>>(p);
    return check_launch("gat_fused_layer_fp8");
}

template <typename T>
static gat_status_t launch_fp8(Fp8Params p, bool fast, int V, cudaStream_t s) {
    if (fast && V == 1) return launch_fp8_fast<T, 1>(p, s);
    if (fast && V == 2) return launch_fp8_fast<T, 2>(p, s);
    p.n_chunks = 0;
    p.heavy_threshold = INT_MAX;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_fp8_generic_kernel<T>,
                                                      kFp8Threads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t wpb = kFp8Threads / 32;
    int64_t blocks = (p.n_rows + wpb - 1) / wpb;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    if (blocks > cap) blocks = cap;
    fused_fp8_generic_kernel<T><<<(unsigned)blocks, kFp8Threads, 0, s>>>(p);
    return check_launch("gat_fused_layer_fp8 (scalar)");
}

}  // namespace gat

using namespace gat;

extern "C" gat_status_t gat_quantize_fp8(const void *x, gat_dtype_t dtype, int64_t n, int32_t H,
                                         int32_t Dh, uint8_t *codes, float *scales, void *stream) {
    if (n < 0 || H < 1 || Dh < 1)
        return fail(GAT_ERR_INVALID_ARG, "gat_quantize_fp8: bad sizes");
    if (dtype != GAT_F32 && dtype != GAT_BF16)
        return fail(GAT_ERR_UNSUPPORTED, "gat_quantize_fp8: unknown dtype %d", (int)dtype);
    if (n == 0) return GAT_OK;
    if (!x || !codes || !scales) return fail(GAT_ERR_INVALID_ARG, "gat_quantize_fp8: NULL pointer");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t cap = (int64_t)sm_count() * 8;
    const int VE = dtype == GAT_F32 ? 4 : 8;
    const int G = Dh / VE;
    if (Dh % VE == 0 && G <= 32 && (G & (G - 1)) == 0 && aligned16(x) &&
        (reinterpret_cast<uintptr_t>(codes) % VE) == 0) {
        int64_t blocks = (n + 7) / 8;
        if (blocks > cap) blocks = cap;
        if (dtype == GAT_F32)
            quantize_fp8_vec_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(
                static_cast<const float *>(x), n, H, Dh, codes, scales);
        else
            quantize_fp8_vec_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
                static_cast<const __nv_bfloat16 *>(x), n, H, Dh, codes, scales);
        return check_launch("gat_quantize_fp8");
    }
    int64_t blocks = (n * H + 7) / 8;
    if (blocks > cap) blocks = cap;
    if (dtype == GAT_F32)
        quantize_fp8_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const float *>(x), n,
                                                                    H, Dh, codes, scales);
    else
        quantize_fp8_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(x), n, H, Dh, codes, scales);
    return check_launch("gat_quantize_fp8");
}

extern "C" gat_status_t gat_fused_layer_fp8(const int32_t *row_ptr, const int32_t *col_idx,
                                            int64_t n_rows, int64_t n_src, int64_t n_edges,
                                            int32_t H, int32_t Dh, float scale, const void *q,
                                            gat_dtype_t dtype, const uint8_t *k8,
                                            const float *k_scale, const uint8_t *v8,
                                            const float *v_scale, void *out, gat_plan_t plan,
                                            void *workspace, size_t workspace_bytes,
                                            void *stream) {
    if (n_rows < 0 || n_src < 0 || n_edges < 0 || H < 1 || Dh < 1)
        return fail(GAT_ERR_INVALID_ARG, "gat_fused_layer_fp8: bad sizes");
    if (dtype != GAT_F32 && dtype != GAT_BF16)
        return fail(GAT_ERR_UNSUPPORTED, "gat_fused_layer_fp8: unknown dtype %d", (int)dtype);
    if (Dh > 256) return fail(GAT_ERR_UNSUPPORTED, "gat_fused_layer_fp8: Dh=%d > 256", (int)Dh);
    if (n_rows == 0) return GAT_OK;
    if (!row_ptr || !q || !out || (n_edges > 0 && (!col_idx || !k8 || !v8 || !k_scale || !v_scale)))
        return fail(GAT_ERR_INVALID_ARG, "gat_fused_layer_fp8: NULL pointer");
    if (plan && (plan->n_rows != n_rows || plan->n_edges != n_edges))
        return fail(GAT_ERR_PLAN_MISMATCH,
                    "gat_fused_layer_fp8: plan is for n_rows=%lld n_edges=%lld",
                    (long long)plan->n_rows, (long long)plan->n_edges);
    Fp8Params p{};
    p.row_ptr = row_ptr;
    p.col_idx = col_idx;
    p.q = q;
    p.k8 = k8;
    p.v8 = v8;
    p.ks = k_scale;
    p.vs = v_scale;
    p.out = out;
    p.n_rows = n_rows;
    p.H = H;
    p.Dh = Dh;
    p.Hs = H;
    p.qscale = scale * kLog2e8;
    p.heavy_threshold = INT_MAX;
    p.slot_floats = slot_floats(H, Dh);
    // vector path: rows of 512 or 1024 codes (32 or 64 16-byte vectors), a
    // head a power-of-two number of whole vectors; wider rows as groups of
    // heads of that size (the widest group dividing H), one launch each
    const int G = Dh / 16;
    int Hg = 0;
    if (Dh % 16 == 0 && (G & (G - 1)) == 0)
        for (int g = H; g >= 1 && !Hg; --g)
            if (H % g == 0 && ((int64_t)g * Dh == 512 || (int64_t)g * Dh == 1024)) Hg = g;
    const bool fast = Hg > 0 && aligned16(q) && aligned16(out) &&
                      (n_edges == 0 || (aligned16(k8) && aligned16(v8)));
    const int V = fast ? (int)((int64_t)Hg * Dh / 512) : 1;
    if (plan && fast) {
        p.heavy_threshold = plan->heavy_threshold;
        p.n_chunks = plan->n_chunks;
        p.chunk_desc = plan->chunk_desc;
        p.chunk_start = plan->chunk_start;
        p.counters = plan->counters;
        if (p.n_chunks > 0) {
            const size_t need = (size_t)p.n_chunks * (size_t)p.slot_floats * sizeof(float);
            if (!workspace || workspace_bytes < need || !aligned16(workspace))
                return fail(GAT_ERR_WORKSPACE,
                            "gat_fused_layer_fp8: workspace needs %zu bytes (16-byte aligned), got %zu",
                            need, workspace_bytes);
            p.partials = static_cast<float *>(workspace);
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fast && Hg < H) {
        // the slices at head h0 of every row: q/out rows (16-byte multiples
        // of Dh elements), code rows (Dh bytes, a multiple of 16) and scale
        // rows; the chunk states of a group fit the workspace sized for H
        const int eb = dtype == GAT_F32 ? 4 : 2;
        for (int h0 = 0; h0 < H; h0 += Hg) {
            Fp8Params pg = p;
            pg.H = Hg;
            pg.q = static_cast<const char *>(q) + (size_t)h0 * Dh * eb;
            pg.out = static_cast<char *>(out) + (size_t)h0 * Dh * eb;
            if (n_edges > 0) {
                pg.k8 = k8 + (size_t)h0 * Dh;
                pg.v8 = v8 + (size_t)h0 * Dh;
                pg.ks = k_scale + h0;
                pg.vs = v_scale + h0;
            }
            const gat_status_t st = dtype == GAT_F32 ? launch_fp8<float>(pg, true, V, s)
                                                     : launch_fp8<__nv_bfloat16>(pg, true, V, s);
            if (st != GAT_OK) return st;
        }
        return GAT_OK;
    }
    if (dtype == GAT_F32) return launch_fp8<float>(p, fast, V, s);
    return launch_fp8<__nv_bfloat16>(p, fast, V, s);
}
