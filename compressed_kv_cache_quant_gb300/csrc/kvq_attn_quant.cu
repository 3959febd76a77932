// a3 kv_decode_attn_quant: fused dequant -> q.k/sqrt(d) -> online softmax ->
// p.v over the quantized paged cache [OnDevice §3.2; TailorKV §2.2], with the
// context split across CTAs and the partial softmax states merged by
// log-sum-exp in the last CTA of every (sequence, kv head).
//
// One CTA = one (sequence b, kv head g, split): it walks 64-token chunks (one
// K quantization group = four 16-token pages), stages the packed codes and
// scales in shared memory and serves all GQ query heads of the group from
// the same staged codes.  A chunk that holds the unfinished K group reads
// its keys from the fp16 tail buffer.
#include <algorithm>
#include <map>
#include <mutex>

#include "kvq_internal.cuh"

namespace {

constexpr int D = KVQ_HEAD_DIM;
constexpr int PG = KVQ_BLOCK_TOKENS;
constexpr int KG = KVQ_K_GROUP_TOKENS;
constexpr int NT = 128;
constexpr int REC = 4 + D;  // partial record: m, l, pad, pad, o[128]

struct QAttnArgs {
    const uint8_t* k_codes;
    const uint8_t* v_codes;
    const uint32_t* k_sz;
    const uint32_t* v_sz;
    const uint16_t* k_tail;
    int64_t num_blocks;
    const int32_t* bt;
    const int32_t* seq_lens;
    int32_t max_blocks;
    int32_t max_len;
    int32_t H;     // kv heads
    int32_t G;     // V group dims
    const uint16_t* q;
    float* out;
    float* part;
    int32_t* counters;
    KvqWsHeader* hdr;
    int32_t n_splits;
    int32_t cps;   // chunks per split
};

__device__ __forceinline__ float2 unpack_sz(uint32_t w) {
    return make_float2(kvq_h2f((uint16_t)(w & 0xffffu)), kvq_h2f((uint16_t)(w >> 16)));
}

template <int BITS, int GQ>
__global__ void __launch_bounds__(NT) qattn_kernel(QAttnArgs a) {
    constexpr int WPR = 4 * BITS;            // 32-bit words per token row
    constexpr int U4_PAGE = PG * WPR / 4;    // uint4 per page of codes
    __shared__ __align__(16) uint32_t kc[KG * WPR];
    __shared__ __align__(16) uint32_t vc[KG * WPR];
    __shared__ float2 vsz[KG * 4];           // (scale, zero) per token and V group
    __shared__ float2 ksz[D];                // (scale, zero) per channel of the K group
    __shared__ __align__(16) float qf[D * GQ];   // q[c][h]
    __shared__ __align__(16) float ps[KG * GQ];  // p[t][h]
    __shared__ float red[NT / 32][GQ];
    __shared__ float m_run[GQ], l_run[GQ], alpha_s[GQ];
    __shared__ int32_t pages[4];
    __shared__ int is_last;

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.seq_lens[b];
    const int n_full = T / KG;
    const int n_chunks = (T + KG - 1) / KG;
    const int nsplit_b = (n_chunks + a.cps - 1) / a.cps;
    const int Hq = a.H * GQ;
    if (T > a.max_len || T < 0) {
        if (tid == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
        return;
    }
    if (n_chunks == 0) {  // empty sequence: output 0
        if (split == 0)
            for (int i = tid; i < GQ * D; i += NT) a.out[((int64_t)b * Hq + g * GQ) * D + i] = 0.0f;
        return;
    }
    if (split >= nsplit_b) return;
    const int c_begin = split * a.cps;
    const int c_end = min(n_chunks, c_begin + a.cps);
    const int NGV = D / a.G;

    // q of the group's heads as fp32, layout [c][h]
    for (int i = tid; i < GQ * D; i += NT) {
        const int h = i / D, c = i % D;
        qf[c * GQ + h] = kvq_h2f(a.q[((int64_t)b * Hq + g * GQ + h) * D + c]);
    }
    if (tid < GQ) {
        m_run[tid] = -INFINITY;
        l_run[tid] = 0.0f;
    }
    float o[GQ];
#pragma unroll
    for (int h = 0; h < GQ; ++h) o[h] = 0.0f;

    const int t_loc = tid >> 1;   // token of this thread in the QK phase
    const int half = tid & 1;     // channel half of this thread in the QK phase

    for (int ch = c_begin; ch < c_end; ++ch) {
        const int t0 = ch * KG;
        const int n_tok = min(KG, T - t0);
        const bool packed = ch < n_full;
        const int n_pages = (n_tok + PG - 1) / PG;
        __syncthreads();  // previous chunk fully consumed
        if (tid < 4) {
            int32_t p = 0;
            if (tid < n_pages) {
                p = a.bt[(int64_t)b * a.max_blocks + ch * 4 + tid];
                if (p < 0 || p >= a.num_blocks) {
                    kvq_dev_flag(a.hdr, KVQ_DEV_BAD_PAGE, b);
                    p = 0;
                }
            }
            pages[tid] = p;
        }
        __syncthreads();
        // stage codes and scales of the chunk
        for (int u = tid; u < n_pages * U4_PAGE; u += NT) {
            const int j = u / U4_PAGE, r = u % U4_PAGE;
            const int64_t base = ((int64_t)pages[j] * a.H + g) * PG * WPR;  // in words
            reinterpret_cast<uint4*>(vc)[u] = reinterpret_cast<const uint4*>(a.v_codes)[base / 4 + r];
            if (packed) reinterpret_cast<uint4*>(kc)[u] = reinterpret_cast<const uint4*>(a.k_codes)[base / 4 + r];
        }
        for (int u = tid; u < n_tok * NGV; u += NT) {
            const int t = u / NGV, j = u % NGV;
            const int64_t slot = ((int64_t)pages[t / PG] * a.H + g) * PG + (t % PG);
            vsz[t * NGV + j] = unpack_sz(a.v_sz[slot * NGV + j]);
        }
        if (packed) ksz[tid] = unpack_sz(a.k_sz[((int64_t)pages[0] * a.H + g) * D + tid]);
        __syncthreads();

        // ---- scores: thread (t_loc, half) covers channels [64 half, 64 half + 64)
        float acc[GQ];
#pragma unroll
        for (int h = 0; h < GQ; ++h) acc[h] = 0.0f;
        const bool valid = t_loc < n_tok;
        if (valid) {
            if (packed) {
                const uint32_t* row = kc + t_loc * WPR;
#pragma unroll 8
                for (int c = 64 * half; c < 64 * half + 64; ++c) {
                    const float2 sz = ksz[c];
                    const float kh = fmaf(sz.x, (float)kvq_get_code<BITS>(row, c), sz.y);
#pragma unroll
                    for (int h = 0; h < GQ; ++h) acc[h] = fmaf(qf[c * GQ + h], kh, acc[h]);
                }
            } else {
                const uint16_t* krow = a.k_tail + (((int64_t)b * a.H + g) * KG + t_loc) * D;
#pragma unroll 8
                for (int c = 64 * half; c < 64 * half + 64; ++c) {
                    const float kh = kvq_h2f(krow[c]);
#pragma unroll
                    for (int h = 0; h < GQ; ++h) acc[h] = fmaf(qf[c * GQ + h], kh, acc[h]);
                }
            }
        }
        float s[GQ];
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 1);
            s[h] = valid ? acc[h] * KVQ_SCORE_LOG2_SCALE : -INFINITY;
            const float wm = kvq_warp_max(s[h]);
            if (lane == 0) red[warp][h] = wm;
        }
        __syncthreads();
        if (tid < GQ) {
            float cm = red[0][tid];
            for (int w = 1; w < NT / 32; ++w) cm = fmaxf(cm, red[w][tid]);
            const float m_new = fmaxf(m_run[tid], cm);
            alpha_s[tid] = exp2f(m_run[tid] - m_new);
            m_run[tid] = m_new;
        }
        __syncthreads();
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            const float p = valid ? exp2f(s[h] - m_run[h]) : 0.0f;
            if (half == 0 && t_loc < KG) ps[t_loc * GQ + h] = p;
            float ws = kvq_warp_sum(half == 0 ? p : 0.0f);
            if (lane == 0) red[warp][h] = ws;
        }
        __syncthreads();
        if (tid < GQ) {
            float lsum = 0.0f;
            for (int w = 0; w < NT / 32; ++w) lsum += red[w][tid];
            l_run[tid] = l_run[tid] * alpha_s[tid] + lsum;
        }
        // ---- p.v: thread = channel d
        {
            const int d = tid;
            const int jg = d / a.G;
#pragma unroll
            for (int h = 0; h < GQ; ++h) o[h] *= alpha_s[h];
#pragma unroll 4
            for (int t = 0; t < n_tok; ++t) {
                const float2 sz = vsz[t * NGV + jg];
                const float vh = fmaf(sz.x, (float)kvq_get_code<BITS>(vc + t * WPR, d), sz.y);
#pragma unroll
                for (int h = 0; h < GQ; ++h) o[h] = fmaf(ps[t * GQ + h], vh, o[h]);
            }
        }
    }
    __syncthreads();

    // ---- partial state of this split
    const int64_t rec0 = (((int64_t)b * a.H + g) * a.n_splits + split) * GQ;
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
        float* r = a.part + (rec0 + h) * REC;
        if (tid == 0) {
            r[0] = m_run[h];
            r[1] = l_run[h];
        }
        r[4 + tid] = o[h];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(&a.counters[b * a.H + g], 1);
        is_last = (prev == nsplit_b - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // ---- last CTA of (b, g): merge the splits by log-sum-exp
    for (int h = 0; h < GQ; ++h) {
        float M = -INFINITY;
        for (int sp = 0; sp < nsplit_b; ++sp) {
            const float* r = a.part + ((((int64_t)b * a.H + g) * a.n_splits + sp) * GQ + h) * REC;
            M = fmaxf(M, __ldcg(r));
        }
        float Lsum = 0.0f, acc = 0.0f;
        for (int sp = 0; sp < nsplit_b; ++sp) {
            const float* r = a.part + ((((int64_t)b * a.H + g) * a.n_splits + sp) * GQ + h) * REC;
            const float w = exp2f(__ldcg(r) - M);
            Lsum = fmaf(__ldcg(r + 1), w, Lsum);
            acc = fmaf(__ldcg(r + 4 + tid), w, acc);
        }
        a.out[((int64_t)b * Hq + g * GQ + h) * D + tid] = acc / Lsum;
    }
    if (tid == 0) a.counters[b * a.H + g] = 0;
}

// ---------------------------------------------------------------- register-centric kernel
//
// Every warp owns 32-token slices of the CTA's range and keeps its own online
// softmax state.  Scores: one token per lane; the query scaled by the slice's K
// group scale, q'[c][h] = q[h][c] * scale_c, sits in shared memory and reaches
// the 32 lanes of a channel in one broadcast load, so
//   s_t = sum_c q[h][c] zero_c + sum_c q'[c][h] code_t[c].
// Values: a lane owns four channels; p'[t][h] = p_t,h * vscale_t is broadcast per
// token and the zero term sum_t p_t,h vzero_t is accumulated per lane and
// reduced once at the end.

constexpr int NWARP = NT / 32;

template <int BITS, int GQ>
struct Q2Smem {
    float qs[GQ][D];                        // query of the group's heads (fp32)
    float qp[NWARP][D][GQ];                 // per warp: query scaled by the slice's K scales
    uint32_t vrow[NWARP][32][4 * BITS];     // per warp: V codes of its 32 tokens
    float pp[NWARP][32][4][GQ];             // per warp: p * V scale, per token, V group, head
    float m[NWARP][GQ], l[NWARP][GQ];
};

__device__ __forceinline__ uint32_t bfe_u32(uint32_t w, uint32_t pos, uint32_t len) {
    uint32_t r;
    asm("bfe.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(w), "r"(pos), "r"(len));
    return r;
}

// small unsigned integer -> float, exactly (2^23 + code, minus 2^23)
__device__ __forceinline__ float code_f(uint32_t code) { return __uint_as_float(code | 0x4B000000u) - 8388608.0f; }

// (d0, d1) += (a0, a1) * b as one packed fp32 FMA (two IEEE fma operations)
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b) {
    asm("{.reg .b64 rd, ra, rb;\n\t"
        "mov.b64 rd, {%0, %1};\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %4};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rd;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1), "f"(b));
}

template <int GQ>
__device__ __forceinline__ void fma_heads(float* acc, const float* qv, float x) {
    if constexpr (GQ == 1) {
        acc[0] = fmaf(qv[0], x, acc[0]);
    } else {
#pragma unroll
        for (int h = 0; h < GQ; h += 2) fma2(acc[h], acc[h + 1], qv[h], qv[h + 1], x);
    }
}

template <int GQ>
__device__ __forceinline__ void lds_heads(float* dst, const float* src) {
    if constexpr (GQ % 4 == 0) {
#pragma unroll
        for (int h = 0; h < GQ; h += 4) {
            const float4 v = *reinterpret_cast<const float4*>(src + h);
            dst[h] = v.x;
            dst[h + 1] = v.y;
            dst[h + 2] = v.z;
            dst[h + 3] = v.w;
        }
    } else if constexpr (GQ == 2) {
        const float2 v = *reinterpret_cast<const float2*>(src);
        dst[0] = v.x;
        dst[1] = v.y;
    } else {
        dst[0] = src[0];
    }
}

template <int BITS, int GQ>
__global__ void __launch_bounds__(NT) qattn2_kernel(QAttnArgs a) {
    constexpr int WPR = 4 * BITS;
    extern __shared__ __align__(16) unsigned char smraw[];
    Q2Smem<BITS, GQ>& S = *reinterpret_cast<Q2Smem<BITS, GQ>*>(smraw);
    __shared__ int is_last;

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    kvq_pdl_begin();
    const int T = a.seq_lens[b];
    const int n_full = T / KG;
    const int n_chunks = (T + KG - 1) / KG;
    const int nsplit_b = (n_chunks + a.cps - 1) / a.cps;
    const int Hq = a.H * GQ;
    if (T > a.max_len || T < 0) {
        if (tid == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
        return;
    }
    if (n_chunks == 0) {  // empty sequence: output 0
        if (split == 0)
            for (int i = tid; i < GQ * D; i += NT) a.out[((int64_t)b * Hq + g * GQ) * D + i] = 0.0f;
        return;
    }
    if (split >= nsplit_b) return;
    const int t_begin = split * a.cps * KG;
    const int t_end = min(T, t_begin + a.cps * KG);
    const int NGV = D / a.G;
    const int jd = (4 * lane) / a.G;  // V group of this lane's four channels
    const int64_t kvrow = (int64_t)b * a.H + g;

    for (int i = tid; i < GQ * D; i += NT) S.qs[i / D][i % D] = kvq_h2f(a.q[((int64_t)b * Hq + g * GQ) * D + i]);
    __syncthreads();

    float m[GQ], l[GQ], o[4][GQ], zt[4][GQ];
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o[i][h] = 0.0f;
            zt[i][h] = 0.0f;
        }
    }
    float(*qp)[GQ] = S.qp[warp];
    for (int s0 = t_begin + 32 * warp; s0 < t_end; s0 += 32 * NWARP) {  // uniform over the warp
        const int t = s0 + lane;
        const bool valid = t < t_end;
        const int gi = s0 / KG;
        const bool packed = gi < n_full;
        int32_t page = 0;
        if (valid) {
            page = a.bt[(int64_t)b * a.max_blocks + (t >> 4)];
            if (page < 0 || page >= a.num_blocks) {
                kvq_dev_flag(a.hdr, KVQ_DEV_BAD_PAGE, b);
                page = 0;
            }
        }
        const int64_t slot = ((int64_t)page * a.H + g) * PG + (t & 15);
        uint32_t kc[WPR];
#pragma unroll
        for (int w = 0; w < WPR; ++w) kc[w] = 0u;
        uint4* vdst = reinterpret_cast<uint4*>(S.vrow[warp][lane]);
#pragma unroll
        for (int u = 0; u < WPR / 4; ++u) {
            uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = make_uint4(0u, 0u, 0u, 0u);
            if (valid) {
                vv = __ldg(reinterpret_cast<const uint4*>(a.v_codes) + slot * (WPR / 4) + u);
                if (packed) kv = __ldg(reinterpret_cast<const uint4*>(a.k_codes) + slot * (WPR / 4) + u);
            }
            kc[4 * u] = kv.x;
            kc[4 * u + 1] = kv.y;
            kc[4 * u + 2] = kv.z;
            kc[4 * u + 3] = kv.w;
            vdst[u] = vv;
        }
        float2 vsz[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            vsz[j] = make_float2(0.f, 0.f);
            if (valid && j < NGV) vsz[j] = unpack_sz(a.v_sz[slot * NGV + j]);
        }
        // query scaled by the K scales of group gi (or plain, for the fp16 tail)
        float c0[GQ];
#pragma unroll
        for (int h = 0; h < GQ; ++h) c0[h] = 0.0f;
        if (packed) {
            int32_t pg = a.bt[(int64_t)b * a.max_blocks + gi * 4];
            if (pg < 0 || pg >= a.num_blocks) {
                kvq_dev_flag(a.hdr, KVQ_DEV_BAD_PAGE, b);
                pg = 0;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = lane + 32 * i;
                const float2 sz = unpack_sz(a.k_sz[((int64_t)pg * a.H + g) * D + c]);
#pragma unroll
                for (int h = 0; h < GQ; ++h) {
                    qp[c][h] = S.qs[h][c] * sz.x;
                    c0[h] = fmaf(S.qs[h][c], sz.y, c0[h]);
                }
            }
#pragma unroll
            for (int h = 0; h < GQ; ++h) c0[h] = kvq_warp_sum(c0[h]);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = lane + 32 * i;
#pragma unroll
                for (int h = 0; h < GQ; ++h) qp[c][h] = S.qs[h][c];
            }
        }
        __syncwarp();
        float sc[GQ];
#pragma unroll
        for (int h = 0; h < GQ; ++h) sc[h] = c0[h];
        if (packed) {
#pragma unroll
            for (int w = 0; w < WPR; ++w) {
                const uint32_t word = kc[w];
#pragma unroll
                for (int i = 0; i < 32 / BITS; ++i) {
                    const int c = w * (32 / BITS) + i;
                    float qv[GQ];
                    lds_heads<GQ>(qv, qp[c]);
                    fma_heads<GQ>(sc, qv, code_f(bfe_u32(word, i * BITS, BITS)));
                }
            }
        } else if (valid) {
            const uint16_t* kr = a.k_tail + (kvrow * KG + (t & (KG - 1))) * D;
            for (int c8 = 0; c8 < D; c8 += 8) {
                const uint4 raw = __ldg(reinterpret_cast<const uint4*>(kr + c8));
                const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 kk = __half22float2(*reinterpret_cast<const __half2*>(&w4[i]));
                    float qv[GQ];
                    lds_heads<GQ>(qv, qp[c8 + 2 * i]);
                    fma_heads<GQ>(sc, qv, kk.x);
                    lds_heads<GQ>(qv, qp[c8 + 2 * i + 1]);
                    fma_heads<GQ>(sc, qv, kk.y);
                }
            }
        }
        // online softmax per head over the warp's 32 tokens
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            const float sh = valid ? sc[h] * KVQ_SCORE_LOG2_SCALE : -INFINITY;
            const float mn = fmaxf(m[h], kvq_warp_max(sh));
            const float alpha = exp2f(m[h] - mn);
            const float p = valid ? exp2f(sh - mn) : 0.0f;
            l[h] = l[h] * alpha + kvq_warp_sum(p);
            m[h] = mn;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                o[i][h] *= alpha;
                zt[i][h] *= alpha;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j < NGV) {
                    S.pp[warp][lane][j][h] = p * vsz[j].x;
                    zt[j][h] = fmaf(p, vsz[j].y, zt[j][h]);
                }
            }
        }
        __syncwarp();
        // values: this lane's channels 4*lane .. 4*lane+3 over the 32 tokens
        const int n_tok = min(32, t_end - s0);
        for (int tt = 0; tt < n_tok; ++tt) {
            float pv[GQ];
            lds_heads<GQ>(pv, S.pp[warp][tt][jd]);
            const uint32_t w = S.vrow[warp][tt][(4 * lane * BITS) >> 5];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float x = code_f(bfe_u32(w, ((4 * lane + i) * BITS) & 31, BITS));
                fma_heads<GQ>(o[i], pv, x);
            }
        }
        __syncwarp();
    }
    // zero term: sum over the warp's lanes of sum_t p vzero, for this lane's V group
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int h = 0; h < GQ; ++h) zt[j][h] = kvq_warp_sum(zt[j][h]);
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
        float z = zt[0][h];
#pragma unroll
        for (int j = 1; j < 4; ++j)
            if (j == jd) z = zt[j][h];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i][h] += z;
    }
    // merge the warps of the CTA (the per-warp query buffers hold the values)
    __syncthreads();
    float* ro = &S.qp[0][0][0];  // [NWARP][GQ][D]
    if (lane == 0)
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            S.m[warp][h] = m[h];
            S.l[warp][h] = l[h];
        }
#pragma unroll
    for (int h = 0; h < GQ; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) ro[(warp * GQ + h) * D + 4 * lane + i] = o[i][h];
    __syncthreads();
    const int64_t rec0 = (((int64_t)b * a.H + g) * a.n_splits + split) * GQ;
    for (int e = tid; e < GQ * D; e += NT) {
        const int h = e / D, d = e % D;
        float M = -INFINITY;
        for (int w = 0; w < NWARP; ++w) M = fmaxf(M, S.m[w][h]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
            for (int w = 0; w < NWARP; ++w) {
                const float wt = exp2f(S.m[w][h] - M);
                L = fmaf(S.l[w][h], wt, L);
                O = fmaf(ro[(w * GQ + h) * D + d], wt, O);
            }
        }
        float* r = a.part + (rec0 + h) * REC;
        if (d == 0) {
            r[0] = M;
            r[1] = L;
        }
        r[4 + d] = O;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(&a.counters[b * a.H + g], 1);
        is_last = (prev == nsplit_b - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // ---- last CTA of (b, g): merge the splits by log-sum-exp
    for (int e = tid; e < GQ * D; e += NT) {
        const int h = e / D, d = e % D;
        float M = -INFINITY;
        for (int sp = 0; sp < nsplit_b; ++sp)
            M = fmaxf(M, __ldcg(a.part + ((((int64_t)b * a.H + g) * a.n_splits + sp) * GQ + h) * REC));
        float Lsum = 0.0f, acc = 0.0f;
        if (M != -INFINITY) {
            for (int sp = 0; sp < nsplit_b; ++sp) {
                const float* r = a.part + ((((int64_t)b * a.H + g) * a.n_splits + sp) * GQ + h) * REC;
                const float w = exp2f(__ldcg(r) - M);
                Lsum = fmaf(__ldcg(r + 1), w, Lsum);
                acc = fmaf(__ldcg(r + 4 + d), w, acc);
            }
        }
        a.out[((int64_t)b * Hq + g * GQ + h) * D + d] = Lsum > 0.0f ? acc / Lsum : 0.0f;
    }
    if (tid == 0) a.counters[b * a.H + g] = 0;
}

struct Plan {
    int n_splits;
    int cps;
};

Plan plan_splits(const kvq_layout* L, const kvq_seqs* S) {
    const int n_chunks = (std::max(S->max_len, 1) + KG - 1) / KG;
    const int64_t units = (int64_t)std::max(S->batch, 1) * L->n_kv_heads;
    const int64_t target = 8LL * kvq_num_sms();  // resident CTAs to aim for
    int splits = (int)std::max<int64_t>(1, (target + units - 1) / units);
    int cps = std::max(4, (n_chunks + splits - 1) / splits);
    cps = std::min(cps, n_chunks);
    splits = (n_chunks + cps - 1) / cps;
    return {splits, cps};
}

size_t ws_layout(const kvq_layout* L, const kvq_seqs* S, size_t* off_part, size_t* off_cnt) {
    const Plan p = plan_splits(L, S);
    const int GQ = L->n_q_heads / L->n_kv_heads;
    const size_t recs = (size_t)std::max(S->batch, 1) * L->n_kv_heads * p.n_splits * GQ;
    *off_part = sizeof(KvqWsHeader);
    *off_cnt = kvq_round_up(*off_part + recs * REC * sizeof(float), 256);
    return kvq_round_up(*off_cnt + (size_t)std::max(S->batch, 1) * L->n_kv_heads * sizeof(int32_t), 256);
}

template <int BITS, int GQ>
int launch_one(dim3 grid, cudaStream_t s, const QAttnArgs& a) {
    const int smem = (int)sizeof(Q2Smem<BITS, GQ>);
    const int st = kvq_prepare_kernel((const void*)qattn2_kernel<BITS, GQ>, smem);
    if (st) return st;
    const cudaError_t e = kvq_launch_pdl(qattn2_kernel<BITS, GQ>, grid, dim3(NT), (size_t)smem, s, a);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_decode_attn_quant launch: %s", cudaGetErrorString(e));
    return KVQ_OK;
}

template <int BITS>
int launch_bits(int gq, dim3 grid, cudaStream_t s, const QAttnArgs& a) {
    switch (gq) {
        case 1: return launch_one<BITS, 1>(grid, s, a);
        case 2: return launch_one<BITS, 2>(grid, s, a);
        case 4: return launch_one<BITS, 4>(grid, s, a);
        default: return launch_one<BITS, 8>(grid, s, a);
    }
}

}  // namespace

extern "C" size_t kv_decode_attn_quant_ws(const kvq_layout* L, const kvq_seqs* S) {
    if (kvq_check_layout(L, "kv_decode_attn_quant_ws", true) || kvq_check_seqs_sizes(S, "kv_decode_attn_quant_ws"))
        return 0;
    size_t a, c;
    return ws_layout(L, S, &a, &c);
}

extern "C" int kv_decode_attn_quant(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q,
                                    float* out, void* ws, size_t ws_bytes, void* stream) {
    kvq_clear_error();
    int st = kvq_check_layout(L, "kv_decode_attn_quant", true);
    if (st) return st;
    st = kvq_check_seqs(S, "kv_decode_attn_quant");
    if (st) return st;
    KVQ_REQUIRE(L->bits != 16, KVQ_ERR_INVALID_ARG, "kv_decode_attn_quant: layer is not quantized (bits == 16)");
    KVQ_REQUIRE(P != nullptr && P->k_codes && P->v_codes && P->k_sz && P->v_sz && P->k_tail, KVQ_ERR_INVALID_ARG,
                "kv_decode_attn_quant: quantized pool arrays missing");
    KVQ_REQUIRE(((uintptr_t)P->k_codes & 15u) == 0 && ((uintptr_t)P->v_codes & 15u) == 0, KVQ_ERR_INVALID_ARG,
                "kv_decode_attn_quant: code arrays must be 16-byte aligned");
    KVQ_REQUIRE(S->batch <= P->max_seqs, KVQ_ERR_INVALID_ARG, "kv_decode_attn_quant: batch exceeds max_seqs");
    size_t off_part, off_cnt;
    const size_t need = ws_layout(L, S, &off_part, &off_cnt);
    st = kvq_check_ws(ws, ws_bytes, need, "kv_decode_attn_quant");
    if (st) return st;
    if (S->batch == 0) return KVQ_OK;
    KVQ_REQUIRE(q && out && S->block_table, KVQ_ERR_INVALID_ARG, "kv_decode_attn_quant: NULL q/out/block table");
    const Plan p = plan_splits(L, S);
    QAttnArgs a;
    a.k_codes = P->k_codes;
    a.v_codes = P->v_codes;
    a.k_sz = reinterpret_cast<const uint32_t*>(P->k_sz);
    a.v_sz = reinterpret_cast<const uint32_t*>(P->v_sz);
    a.k_tail = P->k_tail;
    a.num_blocks = P->num_blocks;
    a.bt = S->block_table;
    a.seq_lens = S->seq_lens;
    a.max_blocks = S->max_blocks;
    a.max_len = S->max_len;
    a.H = L->n_kv_heads;
    a.G = L->v_group_dims;
    a.q = q;
    a.out = out;
    a.part = reinterpret_cast<float*>(static_cast<char*>(ws) + off_part);
    a.counters = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + off_cnt);
    a.hdr = static_cast<KvqWsHeader*>(ws);
    a.n_splits = p.n_splits;
    a.cps = p.cps;
    const int gq = L->n_q_heads / L->n_kv_heads;
    dim3 grid(p.n_splits, L->n_kv_heads, S->batch);
    cudaStream_t s = kvq_stream(stream);
    switch (L->bits) {
        case 1: st = launch_bits<1>(gq, grid, s, a); break;
        case 2: st = launch_bits<2>(gq, grid, s, a); break;
        case 4: st = launch_bits<4>(gq, grid, s, a); break;
        default: st = launch_bits<8>(gq, grid, s, a); break;
    }
    if (st) return st;
    return kvq_launch_status("kv_decode_attn_quant");
}

// ---------------------------------------------------------------- allocation-free variant
//
// For callers that may not reserve device memory of their own: a plugin that
// only receives input and output buffers from a host framework owning every
// allocation, or a latency-critical decode loop that must not enter the CUDA
// allocator (cudaMalloc can synchronize the device and stall other streams).
// The split-K partial states and counters live in one fixed array in the
// library's device image instead of a caller workspace.

#define KVQ_NOALLOC_SCRATCH_BYTES (8u << 20)

static __device__ __align__(256) unsigned char g_qattn_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

// Device address of g_qattn_scratch for the current device, looked up once per
// device (the host-side name of the array is not a device address).
static int qattn_scratch(void** out) {
    static std::mutex mu;
    static std::map<int, void*> addr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_decode_attn_quant_noalloc: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lk(mu);
    auto it = addr.find(dev);
    if (it == addr.end()) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_qattn_scratch);
        if (e != cudaSuccess || p == nullptr)
            return kvq_fail(KVQ_ERR_CUDA, "kv_decode_attn_quant_noalloc: scratch address: %s", cudaGetErrorString(e));
        it = addr.emplace(dev, p).first;
    }
    *out = it->second;
    return KVQ_OK;
}

extern "C" size_t kv_decode_attn_quant_noalloc_max_scratch(void) { return KVQ_NOALLOC_SCRATCH_BYTES; }

extern "C" int kv_decode_attn_quant_noalloc(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S,
                                            const uint16_t* q, float* out, void* stream) {
    kvq_clear_error();
    int st = kvq_check_layout(L, "kv_decode_attn_quant_noalloc", true);
    if (st) return st;
    st = kvq_check_seqs(S, "kv_decode_attn_quant_noalloc");
    if (st) return st;
    KVQ_REQUIRE(L->bits != 16, KVQ_ERR_INVALID_ARG, "kv_decode_attn_quant_noalloc: layer is not quantized");
    KVQ_REQUIRE(P != nullptr && P->k_codes && P->v_codes && P->k_sz && P->v_sz && P->k_tail, KVQ_ERR_INVALID_ARG,
                "kv_decode_attn_quant_noalloc: quantized pool arrays missing");
    KVQ_REQUIRE(((uintptr_t)P->k_codes & 15u) == 0 && ((uintptr_t)P->v_codes & 15u) == 0, KVQ_ERR_INVALID_ARG,
                "kv_decode_attn_quant_noalloc: code arrays must be 16-byte aligned");
    KVQ_REQUIRE(S->batch <= P->max_seqs, KVQ_ERR_INVALID_ARG, "kv_decode_attn_quant_noalloc: batch exceeds max_seqs");
    size_t off_part, off_cnt;
    const size_t need = ws_layout(L, S, &off_part, &off_cnt);
    KVQ_REQUIRE(need <= KVQ_NOALLOC_SCRATCH_BYTES, KVQ_ERR_NO_SPACE,
                "kv_decode_attn_quant_noalloc: this batch needs %zu bytes of scratch, the built-in array holds %u; "
                "use kv_decode_attn_quant with a workspace", need, KVQ_NOALLOC_SCRATCH_BYTES);
    if (S->batch == 0) return KVQ_OK;
    KVQ_REQUIRE(q && out && S->block_table, KVQ_ERR_INVALID_ARG,
                "kv_decode_attn_quant_noalloc: NULL q/out/block table");
    void* ws = nullptr;
    st = qattn_scratch(&ws);
    if (st) return st;
    cudaStream_t s = kvq_stream(stream);
    // The array keeps whatever the previous call left: the status word and the
    // split counters must start at zero.
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(KvqWsHeader), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(static_cast<char*>(ws) + off_cnt, 0, need - off_cnt, s);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_decode_attn_quant_noalloc: %s", cudaGetErrorString(e));
    const Plan p = plan_splits(L, S);
    QAttnArgs a;
    a.k_codes = P->k_codes;
    a.v_codes = P->v_codes;
    a.k_sz = reinterpret_cast<const uint32_t*>(P->k_sz);
    a.v_sz = reinterpret_cast<const uint32_t*>(P->v_sz);
    a.k_tail = P->k_tail;
    a.num_blocks = P->num_blocks;
    a.bt = S->block_table;
    a.seq_lens = S->seq_lens;
    a.max_blocks = S->max_blocks;
    a.max_len = S->max_len;
    a.H = L->n_kv_heads;
    a.G = L->v_group_dims;
    a.q = q;
    a.out = out;
    a.part = reinterpret_cast<float*>(static_cast<char*>(ws) + off_part);
    a.counters = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + off_cnt);
    a.hdr = static_cast<KvqWsHeader*>(ws);
    a.n_splits = p.n_splits;
    a.cps = p.cps;
    const int gq = L->n_q_heads / L->n_kv_heads;
    dim3 grid(p.n_splits, L->n_kv_heads, S->batch);
    switch (L->bits) {
        case 1: st = launch_bits<1>(gq, grid, s, a); break;
        case 2: st = launch_bits<2>(gq, grid, s, a); break;
        case 4: st = launch_bits<4>(gq, grid, s, a); break;
        default: st = launch_bits<8>(gq, grid, s, a); break;
    }
    if (st) return st;
    return kvq_launch_status("kv_decode_attn_quant_noalloc");
}
