// The sparse-layer path [TailorKV §2.3; KVSurvey §三.1; Meeting §3.2, §8.1]:
//   a4 kv_critical_score : s_c = |q_c| max|K_c| -> n_crit channels -> a_t over all tokens
//   a5 kv_topk_select    : sinks + window + top-k by a_t (radix select, cluster of 8 CTAs)
//   a6 kv_sparse_attn    : exact softmax attention over the selected fp16 rows
#include <cooperative_groups.h>

#include <algorithm>

#include "kvq_internal.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int D = KVQ_HEAD_DIM;
constexpr int PG = KVQ_BLOCK_TOKENS;

__device__ __forceinline__ void unpack8(const uint4& r, float* f) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = kvq_h2f((uint16_t)(w[i] & 0xffffu));
        f[2 * i + 1] = kvq_h2f((uint16_t)(w[i] >> 16));
    }
}

// Exclusive scan over the CTA of one uint32 per thread; *total receives the sum.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wsum, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < NT / 32 ? wsum[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NT / 32) wsum[lane] = w;  // inclusive warp prefix
    }
    __syncthreads();
    *total = wsum[NT / 32 - 1];
    return x - v + (warp > 0 ? wsum[warp - 1] : 0u);
}

// ================================================================ a4 critical score (+ fused fp16 append)
//
// A persistent grid: every CTA takes a contiguous run of work items
// (sequence, q head, 2048-token tile), so each CTA meets few heads and
// picks their critical channels once per head.

constexpr int CS_NT = 256;
constexpr int CS_TOK = 8;                          // tokens per thread and item
constexpr int CS_TILE = CS_NT * CS_TOK;            // tokens per work item
constexpr int CS_H1 = 4096;                        // histogram of key bits 31..20
constexpr int CS_MINB = 4;                         // CTAs per SM the grid is sized for
constexpr int CS_BATCH = 8;                        // channel rows loaded before any arithmetic

struct CritArgs {
    uint16_t* kT;
    float* absmax;
    int32_t t_cap;
    const int32_t* seq_lens;
    int32_t max_len;
    int32_t H, GQ;
    const uint16_t* q;
    int32_t n_crit;
    int32_t* crit;
    float* scores;
    int64_t score_stride;
    int32_t tiles;      // work items per (sequence, q head)
    int32_t n_items;    // batch * H_q * tiles
    // fused append of the newest token (k_new == NULL: no append)
    const uint16_t* k_new;
    const uint16_t* v_new;
    uint16_t* k16;
    uint16_t* v16;
    int64_t num_blocks;
    const int32_t* bt;
    int32_t max_blocks;
    // histogram of candidate keys for the selection (NULL: none)
    uint32_t* hist;
    int32_t n_sink, window;
    KvqWsHeader* hdr;
};

__device__ __forceinline__ void unpack8h(const uint4& r, float* f) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}

__global__ void __launch_bounds__(CS_NT, CS_MINB) crit_score_kernel(CritArgs a) {
    __shared__ float sc[D];
    __shared__ float qs[D];
    __shared__ uint16_t knew[D];
    __shared__ int32_t clist[D];
    __shared__ uint32_t lhist[CS_H1];
    const int tid = threadIdx.x;
    const int Hq = a.H * a.GQ;
    const int i_begin = (int)(((int64_t)a.n_items * blockIdx.x) / gridDim.x);
    const int i_end = (int)(((int64_t)a.n_items * (blockIdx.x + 1)) / gridDim.x);
    int cur = -1;  // (sequence, q head) row whose channels and histogram are held
    int T = 0, p_new = -1, cand_lo = 0, cand_hi = 0;
    if (a.hist != nullptr)
        for (int i = tid; i < CS_H1; i += CS_NT) lhist[i] = 0u;
    for (int item = i_begin; item < i_end; ++item) {
        const int rowi = item / a.tiles, tile = item % a.tiles;
        const int b = rowi / Hq, h = rowi % Hq, g = h / a.GQ;
        const int64_t kvrow = (int64_t)b * a.H + g;
        if (rowi != cur) {
            __syncthreads();  // the previous row's channels and histogram are no longer read
            if (a.hist != nullptr && cur >= 0) {
                uint32_t* gh = a.hist + (int64_t)cur * CS_H1;
                for (int i = tid; i < CS_H1; i += CS_NT) {
                    const uint32_t v = lhist[i];
                    if (v) {
                        atomicAdd(&gh[i], v);
                        lhist[i] = 0u;
                    }
                }
            }
            cur = rowi;
            T = a.seq_lens[b];
            if (T < 0 || T > a.max_len || T > a.t_cap) {  // lengths past the buffers are cut and reported
                if (tid == 0 && tile == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
                T = max(0, min(T, min(a.t_cap, a.max_len)));
            }
            p_new = a.k_new != nullptr ? T - 1 : -1;
            cand_lo = a.n_sink;
            cand_hi = T - a.window;
            if (tid < D) {
                const float qv = kvq_h2f(a.q[(int64_t)rowi * D + tid]);
                float am = a.absmax[kvrow * D + tid];
                if (p_new >= 0) {
                    const uint16_t kn = a.k_new[kvrow * D + tid];
                    knew[tid] = kn;
                    am = fmaxf(am, fabsf(kvq_h2f(kn)));
                }
                qs[tid] = qv;
                // |q_c| * max|K_c|: both fp16 values, so the fp32 product is exact
                sc[tid] = fabsf(qv) * am;
            }
            __syncthreads();
            if (tid < 32) {
                // The n_crit largest (s_c, -c): the largest threshold T with at least n_crit
                // composites v_c = key(s_c) << 8 | (255 - c) >= T, found bit by bit.  The
                // composites are distinct, so exactly n_crit channels reach T.
                unsigned long long v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = tid + 32 * j;
                    v[j] = ((unsigned long long)kvq_float_key(sc[c]) << 8) | (unsigned)(255 - c);
                }
                unsigned long long thr = 0ull;
                for (int bit = 39; bit >= 0; --bit) {
                    const unsigned long long t = thr | (1ull << bit);
                    unsigned cnt = 0;
#pragma unroll
                    for (int j = 0; j < 4; ++j) cnt += v[j] >= t;
                    if ((int)__reduce_add_sync(0xffffffffu, cnt) >= a.n_crit) thr = t;
                }
                // list the chosen channels in ascending order
                int before = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool sel = v[j] >= thr;
                    const uint32_t m = __ballot_sync(0xffffffffu, sel);
                    if (sel) clist[before + __popc(m & ((1u << tid) - 1u))] = tid + 32 * j;
                    before += __popc(m);
                }
            }
            __syncthreads();
        }
        if (tile == 0) {
            if (a.crit != nullptr && tid < a.n_crit) a.crit[(int64_t)rowi * a.n_crit + tid] = clist[tid];
            if (p_new >= 0 && h % a.GQ == 0 && tid < D) {
                // append the newest token of kv head g: fp16 rows, channel-major copy, running absmax
                const uint16_t kn = knew[tid];
                const int32_t page = a.bt[(int64_t)b * a.max_blocks + (p_new >> 4)];
                if (page >= 0 && page < a.num_blocks) {
                    const int64_t off = ((page * (int64_t)a.H + g) * PG + (p_new & 15)) * D + tid;
                    a.k16[off] = kn;
                    a.v16[off] = a.v_new[kvrow * D + tid];
                } else {
                    kvq_dev_flag(a.hdr, KVQ_DEV_BAD_PAGE, b);
                }
                a.kT[(kvrow * D + tid) * a.t_cap + p_new] = kn;
                a.absmax[kvrow * D + tid] = fmaxf(a.absmax[kvrow * D + tid], fabsf(kvq_h2f(kn)));
            }
        }
        const int t0 = tile * CS_TILE + tid * CS_TOK;
        if (t0 >= T) continue;
        const uint16_t* base = a.kT + kvrow * D * a.t_cap + t0;
        float acc[CS_TOK];
#pragma unroll
        for (int i = 0; i < CS_TOK; ++i) acc[i] = 0.0f;
        for (int j0 = 0; j0 < a.n_crit; j0 += CS_BATCH) {
            // all loads of the batch in flight before the arithmetic
            uint4 raw[CS_BATCH];
#pragma unroll
            for (int j = 0; j < CS_BATCH; ++j)
                if (j0 + j < a.n_crit)
                    raw[j] = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)clist[j0 + j] * a.t_cap));
            const bool has_new = p_new >= t0 && p_new < t0 + CS_TOK;
#pragma unroll
            for (int j = 0; j < CS_BATCH; ++j) {
                if (j0 + j >= a.n_crit) break;
                const int c = clist[j0 + j];  // ascending channel order
                const float qc = qs[c];
                float k[8];
                unpack8h(raw[j], k);
                if (has_new) {
                    // the newest token is taken from k_new: its kT column may be written concurrently
#pragma unroll
                    for (int i = 0; i < CS_TOK; ++i)
                        if (p_new == t0 + i) k[i] = kvq_h2f(knew[c]);
                }
                // fma == add of the exact fp16*fp16 product: the same fp32 result as (q*k) + acc
#pragma unroll
                for (int i = 0; i < CS_TOK; ++i) acc[i] = fmaf(qc, k[i], acc[i]);
            }
        }
        float* out = a.scores + (int64_t)rowi * a.score_stride + t0;
        if (t0 + CS_TOK <= T) {
            reinterpret_cast<float4*>(out)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            reinterpret_cast<float4*>(out)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        } else {
#pragma unroll
            for (int i = 0; i < CS_TOK; ++i)
                if (i < T - t0) out[i] = acc[i];
        }
        if (a.hist != nullptr) {
#pragma unroll
            for (int i = 0; i < CS_TOK; ++i) {
                const int t = t0 + i;
                if (t >= cand_lo && t < cand_hi) atomicAdd(&lhist[kvq_float_key(acc[i]) >> 20], 1u);
            }
        }
    }
    if (a.hist != nullptr && cur >= 0) {
        __syncthreads();
        uint32_t* gh = a.hist + (int64_t)cur * CS_H1;
        for (int i = tid; i < CS_H1; i += CS_NT) {
            const uint32_t v = lhist[i];
            if (v) atomicAdd(&gh[i], v);
        }
    }
}

// ================================================================ a6 sparse attention

constexpr int SA_NT = 256;
constexpr int SA_HW = SA_NT / 16;  // half-warps per CTA
constexpr int SA_BATCH = 4;        // rows in flight per half-warp
constexpr int SA_REC = 4 + D;
constexpr int SA_MAX_RPS = 2048;   // rows per split: their offsets are resolved into shared memory

struct SAArgs {
    const uint16_t* k16;
    const uint16_t* v16;
    int64_t num_blocks;
    const int32_t* bt;
    const int32_t* seq_lens;
    int32_t max_blocks;
    int32_t max_len;
    int32_t H, GQ;
    const uint16_t* q;
    const int32_t* sel;
    int32_t sel_cap;
    const int32_t* sel_count;
    int32_t per_kv;     // lists per kv head
    float* out;
    float* probs;
    float* part;
    int32_t* counters;
    KvqWsHeader* hdr;
    int32_t n_splits;
    int32_t rps;        // rows per split
};

template <int NH>
__global__ void __launch_bounds__(SA_NT) sparse_attn_kernel(SAArgs a) {
    extern __shared__ __align__(16) float sm[];  // [SA_HW][NH][SA_REC] half-warp states
    __shared__ int is_last;
    const int split = blockIdx.x, list = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, hw = tid >> 4, l16 = tid & 15;
    const int n_lists = a.per_kv ? a.H : a.H * a.GQ;
    const int Hq = a.H * a.GQ;
    const int g = a.per_kv ? list : list / a.GQ;
    const int h0 = a.per_kv ? list * a.GQ : list;
    int T = a.seq_lens[b];
    if (T > a.max_len) {  // ids are checked against min(seq_len, max_len): the block table's reach
        if (tid == 0 && split == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
        T = a.max_len;
    }
    int n = a.sel_count[(int64_t)b * n_lists + list];
    if (n > a.sel_cap || n < 0) {
        if (tid == 0 && split == 0) kvq_dev_flag(a.hdr, KVQ_DEV_OVERFLOW, b);
        n = max(0, min(n, a.sel_cap));
    }
    if (n == 0) {
        if (split == 0)
            for (int i = tid; i < NH * D; i += SA_NT) a.out[((int64_t)b * Hq + h0) * D + i] = 0.0f;
        return;
    }
    const int nsplit_b = (n + a.rps - 1) / a.rps;
    if (split >= nsplit_b) return;
    const int r_begin = split * a.rps, r_end = min(n, r_begin + a.rps);
    const int32_t* ids = a.sel + ((int64_t)b * n_lists + list) * a.sel_cap;

    // the split's rows: ids and pages resolved up front into row offsets (in 128-element rows;
    // ~0u for a bad id or page), four per thread in flight
    uint32_t* roff = reinterpret_cast<uint32_t*>(sm + SA_HW * NH * SA_REC);
    for (int i0 = r_begin + tid; i0 < r_end; i0 += 4 * SA_NT) {
        int t[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * SA_NT;
            t[u] = i < r_end ? ids[i] : -1;
        }
        int32_t pg[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            pg[u] = t[u] >= 0 && t[u] < T ? a.bt[(int64_t)b * a.max_blocks + (t[u] >> 4)] : -1;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * SA_NT;
            if (i >= r_end) continue;
            uint32_t r = 0xffffffffu;
            if (t[u] < 0 || t[u] >= T) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_INDEX, t[u]);
            else if (pg[u] < 0 || pg[u] >= a.num_blocks) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_PAGE, t[u]);
            else r = (uint32_t)(((int64_t)pg[u] * a.H + g) * PG + (t[u] & 15));
            roff[i - r_begin] = r;
        }
    }
    __syncthreads();

    float qv[NH][8];
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        const uint4 raw = *reinterpret_cast<const uint4*>(a.q + ((int64_t)b * Hq + h0 + hh) * D + 8 * l16);
        unpack8(raw, qv[hh]);
#pragma unroll
        for (int i = 0; i < 8; ++i) qv[hh][i] *= KVQ_SCORE_LOG2_SCALE;
    }
    float m[NH], l[NH], o[NH][8];
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[hh][i] = 0.0f;
    }
    // The loop bound is uniform over the CTA so that every lane reaches the shuffles.
    for (int it = r_begin; it < r_end; it += SA_HW * SA_BATCH) {
        uint4 kr[SA_BATCH], vr[SA_BATCH];
        bool ok[SA_BATCH];
#pragma unroll
        for (int j = 0; j < SA_BATCH; ++j) {
            const int i = it + j * SA_HW + hw;
            ok[j] = false;
            kr[j] = make_uint4(0u, 0u, 0u, 0u);
            vr[j] = make_uint4(0u, 0u, 0u, 0u);
            const uint32_t r = i < r_end ? roff[i - r_begin] : 0xffffffffu;
            if (r != 0xffffffffu) {
                const int64_t off = (int64_t)r * D + 8 * l16;
                kr[j] = __ldg(reinterpret_cast<const uint4*>(a.k16 + off));
                vr[j] = __ldg(reinterpret_cast<const uint4*>(a.v16 + off));
                ok[j] = true;
            }
        }
        float s[SA_BATCH][NH];
#pragma unroll
        for (int j = 0; j < SA_BATCH; ++j) {
            float kf[8];
            unpack8(kr[j], kf);
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                float acc = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i) acc = fmaf(qv[hh][i], kf[i], acc);
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                s[j][hh] = ok[j] ? acc : -INFINITY;
            }
        }
        if (a.probs != nullptr && l16 == 0) {
#pragma unroll
            for (int j = 0; j < SA_BATCH; ++j) {
                const int i = it + j * SA_HW + hw;
                if (i < r_end)
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh)
                        a.probs[((int64_t)b * Hq + h0 + hh) * a.sel_cap + i] = s[j][hh];
            }
        }
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
            float mn = m[hh];
#pragma unroll
            for (int j = 0; j < SA_BATCH; ++j) mn = fmaxf(mn, s[j][hh]);
            if (mn == -INFINITY) continue;
            const float alpha = exp2f(m[hh] - mn);
            m[hh] = mn;
            l[hh] *= alpha;
#pragma unroll
            for (int i = 0; i < 8; ++i) o[hh][i] *= alpha;
#pragma unroll
            for (int j = 0; j < SA_BATCH; ++j) {
                const float p = exp2f(s[j][hh] - mn);
                l[hh] += p;
                float vf[8];
                unpack8(vr[j], vf);
#pragma unroll
                for (int i = 0; i < 8; ++i) o[hh][i] = fmaf(p, vf[i], o[hh][i]);
            }
        }
    }
    // ---- merge the half-warp states of the CTA
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        float* r = sm + (hw * NH + hh) * SA_REC;
        if (l16 == 0) {
            r[0] = m[hh];
            r[1] = l[hh];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) r[4 + 8 * l16 + i] = o[hh][i];
    }
    __syncthreads();
    const int64_t rec0 = (((int64_t)b * n_lists + list) * a.n_splits + split) * NH;
    for (int e = tid; e < NH * D; e += SA_NT) {
        const int hh = e / D, d = e % D;
        float M = -INFINITY;
        for (int w = 0; w < SA_HW; ++w) M = fmaxf(M, sm[(w * NH + hh) * SA_REC]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
            for (int w = 0; w < SA_HW; ++w) {
                const float* r = sm + (w * NH + hh) * SA_REC;
                const float wt = exp2f(r[0] - M);
                L = fmaf(r[1], wt, L);
                O = fmaf(r[4 + d], wt, O);
            }
        }
        float* dst = a.part + (rec0 + hh) * SA_REC;
        if (d == 0) {
            dst[0] = M;
            dst[1] = L;
        }
        dst[4 + d] = O;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(&a.counters[(int64_t)b * n_lists + list], 1);
        is_last = (prev == nsplit_b - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // ---- last CTA: merge the splits, write the output and normalize the probabilities
    __shared__ float fin_m[8], fin_l[8];
    for (int e = tid; e < NH * D; e += SA_NT) {
        const int hh = e / D, d = e % D;
        float M = -INFINITY;
        for (int sp = 0; sp < nsplit_b; ++sp)
            M = fmaxf(M, __ldcg(a.part + ((((int64_t)b * n_lists + list) * a.n_splits + sp) * NH + hh) * SA_REC));
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
            for (int sp = 0; sp < nsplit_b; ++sp) {
                const float* r = a.part + ((((int64_t)b * n_lists + list) * a.n_splits + sp) * NH + hh) * SA_REC;
                const float wt = exp2f(__ldcg(r) - M);
                L = fmaf(__ldcg(r + 1), wt, L);
                O = fmaf(__ldcg(r + 4 + d), wt, O);
            }
        }
        a.out[((int64_t)b * Hq + h0 + hh) * D + d] = L > 0.0f ? O / L : 0.0f;
        if (d == 0) {
            fin_m[hh] = M;
            fin_l[hh] = L;
        }
    }
    if (tid == 0) a.counters[(int64_t)b * n_lists + list] = 0;
    if (a.probs == nullptr) return;
    __syncthreads();
    // the stored scores become probabilities; every thread keeps 2 x NH loads in flight
    float* pr0 = a.probs + ((int64_t)b * Hq + h0) * a.sel_cap;
    for (int i0 = tid; i0 < n; i0 += 2 * SA_NT) {
        float sv[2][NH];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const int i = i0 + u * SA_NT;
                sv[u][hh] = i < n ? __ldcg(pr0 + (int64_t)hh * a.sel_cap + i) : -INFINITY;
            }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const int i = i0 + u * SA_NT;
                const float M = fin_m[hh], L = fin_l[hh];
                if (i < n) pr0[(int64_t)hh * a.sel_cap + i] = (L > 0.0f && sv[u][hh] != -INFINITY) ? exp2f(sv[u][hh] - M) / L : 0.0f;
            }
    }
}

struct SAPlan {
    int n_splits, rps;
};

SAPlan sa_plan(const kvq_layout* L, const kvq_seqs* S, int32_t sel_cap, int per_kv) {
    const int n_lists = per_kv ? L->n_kv_heads : L->n_q_heads;
    const int64_t units = (int64_t)std::max(S->batch, 1) * n_lists;
    const int64_t target = 3LL * kvq_num_sms();
    int splits = (int)std::max<int64_t>(1, (target + units - 1) / units);
    int rps = (std::max(sel_cap, 1) + splits - 1) / splits;
    rps = std::min(SA_MAX_RPS, std::max(64, (rps + 63) / 64 * 64));
    splits = (std::max(sel_cap, 1) + rps - 1) / rps;
    return {splits, rps};
}

size_t sa_ws_layout(const kvq_layout* L, const kvq_seqs* S, int32_t sel_cap, size_t* off_part, size_t* off_cnt) {
    // sized for the larger of the two list modes so one workspace serves both
    const SAPlan p0 = sa_plan(L, S, sel_cap, 0), p1 = sa_plan(L, S, sel_cap, 1);
    const int GQ = L->n_q_heads / std::max(L->n_kv_heads, 1);
    const size_t r0 = (size_t)std::max(S->batch, 1) * L->n_q_heads * p0.n_splits;
    const size_t r1 = (size_t)std::max(S->batch, 1) * L->n_kv_heads * p1.n_splits * GQ;
    const size_t recs = r0 > r1 ? r0 : r1;
    *off_part = sizeof(KvqWsHeader);
    *off_cnt = kvq_round_up(*off_part + recs * SA_REC * sizeof(float), 256);
    return kvq_round_up(*off_cnt + (size_t)std::max(S->batch, 1) * L->n_q_heads * sizeof(int32_t), 256);
}

template <int NH>
int launch_sa(const SAArgs& a, dim3 grid, cudaStream_t s) {
    const size_t smem = (size_t)SA_HW * NH * SA_REC * sizeof(float) + (size_t)a.rps * sizeof(uint32_t);
    const int st = kvq_prepare_kernel((const void*)sparse_attn_kernel<NH>,
                                      (int)((size_t)SA_HW * NH * SA_REC * sizeof(float) + SA_MAX_RPS * sizeof(uint32_t)));
    if (st) return st;
    sparse_attn_kernel<NH><<<grid, SA_NT, smem, s>>>(a);
    return kvq_launch_status("kv_sparse_attn");
}

}  // namespace

// ================================================================ ABI

namespace {

int crit_common(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q, int32_t n_crit,
                float* scores, int64_t score_stride, const char* fn) {
    int st = kvq_check_layout(L, fn, true);
    if (st) return st;
    st = kvq_check_seqs(S, fn);
    if (st) return st;
    KVQ_REQUIRE(L->bits == 16, KVQ_ERR_INVALID_ARG, "%s: not an fp16 layer", fn);
    KVQ_REQUIRE(P && P->kT && P->k_absmax, KVQ_ERR_INVALID_ARG, "%s: pool needs kT and k_absmax", fn);
    KVQ_REQUIRE(n_crit >= 1 && n_crit <= D, KVQ_ERR_INVALID_ARG, "%s: n_crit %d not in [1, 128]", fn, n_crit);
    KVQ_REQUIRE(P->t_cap % 8 == 0 && P->t_cap >= S->max_len, KVQ_ERR_INVALID_ARG,
                "%s: t_cap must be a multiple of 8 and >= max_len", fn);
    KVQ_REQUIRE(((uintptr_t)P->kT & 15u) == 0, KVQ_ERR_INVALID_ARG, "%s: kT must be 16-byte aligned", fn);
    KVQ_REQUIRE(scores && ((uintptr_t)scores & 15u) == 0 && score_stride % 4 == 0 && score_stride >= S->max_len,
                KVQ_ERR_INVALID_ARG, "%s: scores must be 16-byte aligned, stride %% 4 == 0, >= max_len", fn);
    KVQ_REQUIRE(S->batch <= P->max_seqs, KVQ_ERR_INVALID_ARG, "%s: batch exceeds max_seqs", fn);
    KVQ_REQUIRE(S->batch == 0 || q != nullptr, KVQ_ERR_INVALID_ARG, "%s: NULL q", fn);
    return KVQ_OK;
}

CritArgs crit_args(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q, int32_t n_crit,
                   int32_t* crit, float* scores, int64_t score_stride) {
    CritArgs a{};
    a.kT = P->kT;
    a.absmax = P->k_absmax;
    a.t_cap = P->t_cap;
    a.seq_lens = S->seq_lens;
    a.max_len = S->max_len;
    a.H = L->n_kv_heads;
    a.GQ = L->n_q_heads / L->n_kv_heads;
    a.q = q;
    a.n_crit = n_crit;
    a.crit = crit;
    a.scores = scores;
    a.score_stride = score_stride;
    return a;
}

int launch_crit(CritArgs& a, const kvq_layout* L, const kvq_seqs* S, cudaStream_t s) {
    const int st = kvq_prepare_kernel((const void*)crit_score_kernel, 0);
    if (st) return st;
    a.tiles = std::max(1, (S->max_len + CS_TILE - 1) / CS_TILE);
    a.n_items = S->batch * L->n_q_heads * a.tiles;
    const int grid = std::min(a.n_items, kvq_num_sms() * CS_MINB);
    crit_score_kernel<<<grid, CS_NT, 0, s>>>(a);
    return KVQ_OK;
}

}  // namespace

extern "C" int kv_critical_score(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q,
                                 int32_t n_crit, int32_t* crit, float* scores, int64_t score_stride,
                                 void* stream) {
    kvq_clear_error();
    int st = crit_common(L, P, S, q, n_crit, scores, score_stride, "kv_critical_score");
    if (st) return st;
    if (S->batch == 0) return KVQ_OK;
    CritArgs a = crit_args(L, P, S, q, n_crit, crit, scores, score_stride);
    st = launch_crit(a, L, S, kvq_stream(stream));
    if (st) return st;
    return kvq_launch_status("kv_critical_score");
}

extern "C" size_t kv_append_critical_score_ws(void) { return sizeof(KvqWsHeader); }

extern "C" int kv_append_critical_score(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S,
                                        const uint16_t* k_new, const uint16_t* v_new, const uint16_t* q,
                                        int32_t n_crit, int32_t* crit, float* scores, int64_t score_stride,
                                        uint32_t* hist, int32_t n_sink, int32_t window, void* ws, size_t ws_bytes,
                                        void* stream) {
    kvq_clear_error();
    int st = crit_common(L, P, S, q, n_crit, scores, score_stride, "kv_append_critical_score");
    if (st) return st;
    st = kvq_check_ws(ws, ws_bytes, kv_append_critical_score_ws(), "kv_append_critical_score");
    if (st) return st;
    KVQ_REQUIRE(P->k16 && P->v16, KVQ_ERR_INVALID_ARG, "kv_append_critical_score: pool needs k16 and v16");
    KVQ_REQUIRE(n_sink >= 0 && window >= 0, KVQ_ERR_INVALID_ARG, "kv_append_critical_score: n_sink / window");
    if (S->batch == 0) return KVQ_OK;
    KVQ_REQUIRE(k_new && v_new && S->block_table, KVQ_ERR_INVALID_ARG,
                "kv_append_critical_score: NULL k_new / v_new / block table");
    CritArgs a = crit_args(L, P, S, q, n_crit, crit, scores, score_stride);
    a.k_new = k_new;
    a.v_new = v_new;
    a.k16 = P->k16;
    a.v16 = P->v16;
    a.num_blocks = P->num_blocks;
    a.bt = S->block_table;
    a.max_blocks = S->max_blocks;
    a.hist = hist;
    a.n_sink = n_sink;
    a.window = window;
    a.hdr = static_cast<KvqWsHeader*>(ws);
    st = launch_crit(a, L, S, kvq_stream(stream));
    if (st) return st;
    return kvq_launch_status("kv_append_critical_score");
}

extern "C" size_t kv_sparse_attn_ws(const kvq_layout* L, const kvq_seqs* S, int32_t sel_cap) {
    if (kvq_check_layout(L, "kv_sparse_attn_ws", true) || kvq_check_seqs_sizes(S, "kv_sparse_attn_ws") || sel_cap <= 0)
        return 0;
    size_t a, c;
    return sa_ws_layout(L, S, sel_cap, &a, &c);
}

extern "C" int kv_sparse_attn(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q,
                              const int32_t* sel, int32_t sel_cap, const int32_t* sel_count, int32_t sel_per_kv_head,
                              float* out, float* probs, void* ws, size_t ws_bytes, void* stream) {
    kvq_clear_error();
    int st = kvq_check_layout(L, "kv_sparse_attn", true);
    if (st) return st;
    st = kvq_check_seqs(S, "kv_sparse_attn");
    if (st) return st;
    KVQ_REQUIRE(P && P->k16 && P->v16, KVQ_ERR_INVALID_ARG, "kv_sparse_attn: pool needs k16 and v16");
    KVQ_REQUIRE(((uintptr_t)P->k16 & 15u) == 0 && ((uintptr_t)P->v16 & 15u) == 0, KVQ_ERR_INVALID_ARG,
                "kv_sparse_attn: k16/v16 must be 16-byte aligned");
    KVQ_REQUIRE(sel_cap > 0 && sel && sel_count && out, KVQ_ERR_INVALID_ARG, "kv_sparse_attn: NULL buffer or sel_cap");
    KVQ_REQUIRE(sel_per_kv_head == 0 || sel_per_kv_head == 1, KVQ_ERR_INVALID_ARG, "kv_sparse_attn: sel_per_kv_head");
    size_t off_part, off_cnt;
    const size_t need = sa_ws_layout(L, S, sel_cap, &off_part, &off_cnt);
    st = kvq_check_ws(ws, ws_bytes, need, "kv_sparse_attn");
    if (st) return st;
    if (S->batch == 0) return KVQ_OK;
    KVQ_REQUIRE(q && S->block_table && ((uintptr_t)q & 15u) == 0, KVQ_ERR_INVALID_ARG,
                "kv_sparse_attn: q must be 16-byte aligned; block table needed");
    const SAPlan p = sa_plan(L, S, sel_cap, sel_per_kv_head);
    SAArgs a;
    a.k16 = P->k16;
    a.v16 = P->v16;
    a.num_blocks = P->num_blocks;
    a.bt = S->block_table;
    a.seq_lens = S->seq_lens;
    a.max_blocks = S->max_blocks;
    a.max_len = S->max_len;
    a.H = L->n_kv_heads;
    a.GQ = L->n_q_heads / L->n_kv_heads;
    a.q = q;
    a.sel = sel;
    a.sel_cap = sel_cap;
    a.sel_count = sel_count;
    a.per_kv = sel_per_kv_head;
    a.out = out;
    a.probs = probs;
    a.part = reinterpret_cast<float*>(static_cast<char*>(ws) + off_part);
    a.counters = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + off_cnt);
    a.hdr = static_cast<KvqWsHeader*>(ws);
    a.n_splits = p.n_splits;
    a.rps = p.rps;
    const int n_lists = sel_per_kv_head ? L->n_kv_heads : L->n_q_heads;
    dim3 grid(p.n_splits, n_lists, S->batch);
    cudaStream_t s = kvq_stream(stream);
    if (!sel_per_kv_head) return launch_sa<1>(a, grid, s);
    switch (a.GQ) {
        case 1: return launch_sa<1>(a, grid, s);
        case 2: return launch_sa<2>(a, grid, s);
        case 4: return launch_sa<4>(a, grid, s);
        default: return launch_sa<8>(a, grid, s);
    }
}
