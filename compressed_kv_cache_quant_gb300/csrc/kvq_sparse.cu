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

// ================================================================ a4 critical score

constexpr int CS_NT = 256;
constexpr int CS_TOK = 8;                 // tokens per thread
constexpr int CS_TILE = CS_NT * CS_TOK;   // tokens per CTA

struct CritArgs {
    const uint16_t* kT;
    const float* absmax;
    int32_t t_cap;
    const int32_t* seq_lens;
    int32_t max_len;
    int32_t H, GQ;
    const uint16_t* q;
    int32_t n_crit;
    int32_t* crit;
    float* scores;
    int64_t score_stride;
};

__global__ void __launch_bounds__(CS_NT) crit_score_kernel(CritArgs a) {
    __shared__ float sc[D];
    __shared__ float qs[D];
    __shared__ int32_t clist[D];
    __shared__ uint32_t selmask[D / 32];
    const int tile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const int g = h / a.GQ;
    const int Hq = a.H * a.GQ;
    const int T = max(0, min(a.seq_lens[b], min(a.t_cap, a.max_len)));  // lengths past the buffers are cut
    if (tile > 0 && tile * CS_TILE >= T) return;
    if (tid < D) {
        const float qv = kvq_h2f(a.q[((int64_t)b * Hq + h) * D + tid]);
        qs[tid] = qv;
        // |q_c| * max|K_c|: both fp16 values, so the fp32 product is exact
        sc[tid] = fabsf(qv) * a.absmax[((int64_t)b * a.H + g) * D + tid];
    }
    __syncthreads();
    bool sel = false;
    if (tid < D) {
        const float my = sc[tid];
        int rank = 0;
        for (int c2 = 0; c2 < D; ++c2) {
            const float v = sc[c2];
            rank += (v > my) || (v == my && c2 < tid);
        }
        sel = rank < a.n_crit;
        const uint32_t m = __ballot_sync(0xffffffffu, sel);
        if ((tid & 31) == 0) selmask[tid >> 5] = m;
    }
    __syncthreads();
    if (tid < D && sel) {
        int idx = __popc(selmask[tid >> 5] & ((1u << (tid & 31)) - 1u));
        for (int w = 0; w < (tid >> 5); ++w) idx += __popc(selmask[w]);
        clist[idx] = tid;
    }
    __syncthreads();
    if (tile == 0 && a.crit != nullptr && tid < a.n_crit) a.crit[((int64_t)b * Hq + h) * a.n_crit + tid] = clist[tid];
    const int t0 = (tile * CS_NT + tid) * CS_TOK;
    if (t0 >= T) return;
    float acc[CS_TOK];
#pragma unroll
    for (int i = 0; i < CS_TOK; ++i) acc[i] = 0.0f;
    const uint16_t* base = a.kT + ((int64_t)b * a.H + g) * D * a.t_cap + t0;
#pragma unroll 8
    for (int j = 0; j < a.n_crit; ++j) {
        const int c = clist[j];  // ascending channel order
        const float qc = qs[c];
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)c * a.t_cap));
        float k[8];
        unpack8(raw, k);
        // fma == add of the exact fp16*fp16 product: the same fp32 result as (q*k) + acc
#pragma unroll
        for (int i = 0; i < CS_TOK; ++i) acc[i] = fmaf(qc, k[i], acc[i]);
    }
    float* out = a.scores + ((int64_t)b * Hq + h) * a.score_stride + t0;
    if (t0 + CS_TOK <= T) {
        reinterpret_cast<float4*>(out)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        reinterpret_cast<float4*>(out)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
        for (int i = 0; i < T - t0; ++i) out[i] = acc[i];
    }
}

// ================================================================ a5 top-k select

constexpr int SEL_CL = 8;     // CTAs per cluster: one cluster per (sequence, head)
constexpr int SEL_NT = 512;
constexpr int SEL_MAX_CHUNK = 49152;  // keys per CTA held in shared memory

struct SelArgs {
    const float* scores;
    int64_t score_stride;
    const int32_t* seq_lens;
    int32_t max_len;
    int32_t n_heads;
    int32_t k_fixed;
    double ratio;
    int32_t n_sink;
    int32_t window;
    int32_t* sel;
    int32_t sel_cap;
    int32_t* sel_count;
    KvqWsHeader* hdr;
};

__global__ void __cluster_dims__(SEL_CL, 1, 1) __launch_bounds__(SEL_NT) topk_select_kernel(SelArgs a) {
    extern __shared__ __align__(16) uint32_t keys[];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t tot[256];
    __shared__ uint32_t wsum[SEL_NT / 32];
    __shared__ uint32_t xch[2];
    __shared__ uint32_t s_bin, s_above;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const int T = a.seq_lens[b];
    int32_t* out = a.sel + ((int64_t)b * a.n_heads + h) * a.sel_cap;
    if (T < 0 || T > a.max_len) {  // uniform over the cluster: every CTA leaves here
        if (tid == 0 && rank == 0) {
            kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
            a.sel_count[(int64_t)b * a.n_heads + h] = 0;
        }
        return;
    }
    const int k = a.k_fixed >= 0 ? a.k_fixed : (int)floor(a.ratio * (double)T);
    const int chunk = (T + SEL_CL - 1) / SEL_CL;
    const int lo = min(T, rank * chunk), hi = min(T, lo + chunk);
    if ((int64_t)T <= (int64_t)a.n_sink + a.window + k) {  // everything is kept
        for (int p = lo + tid; p < hi; p += SEL_NT)
            if (p < a.sel_cap) out[p] = p;
        if (rank == 0 && tid == 0) {
            if (T > a.sel_cap) kvq_dev_flag(a.hdr, KVQ_DEV_OVERFLOW, b);
            a.sel_count[(int64_t)b * a.n_heads + h] = min(T, a.sel_cap);
        }
        return;
    }
    const int cand_lo = a.n_sink, cand_hi = T - a.window;
    const float* row = a.scores + ((int64_t)b * a.n_heads + h) * a.score_stride;
    for (int p = lo + tid; p < hi; p += SEL_NT) keys[p - lo] = kvq_float_key(row[p]);

    // ---- radix select of the k-th largest candidate key, 8 bits per pass
    uint32_t prefix = 0u, mask = 0u, remaining = (uint32_t)k;
    if (k > 0) {
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            for (int i = tid; i < 256; i += SEL_NT) hist[i] = 0u;
            __syncthreads();
            for (int p = max(lo, cand_lo) + tid; p < min(hi, cand_hi); p += SEL_NT) {
                const uint32_t key = keys[p - lo];
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            }
            cluster.sync();
            if (tid < 256) {
                uint32_t s = 0;
                for (int r = 0; r < SEL_CL; ++r) s += cluster.map_shared_rank(hist, r)[tid];
                tot[tid] = s;
            }
            cluster.sync();
            if (tid < 32) {
                // lane l owns bins [248 - 8l, 255 - 8l]; lane 0 the largest
                uint32_t ls = 0;
                for (int j = 0; j < 8; ++j) ls += tot[255 - 8 * tid - j];
                uint32_t incl = ls;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (tid >= o) incl += y;
                }
                const uint32_t ballot = __ballot_sync(0xffffffffu, incl >= remaining);
                const int l = __ffs(ballot) - 1;  // first lane reaching `remaining`
                if (tid == l) {
                    uint32_t run = incl - ls;
                    for (int j = 0; j < 8; ++j) {
                        const int bin = 255 - 8 * tid - j;
                        if (run + tot[bin] >= remaining) {
                            s_bin = (uint32_t)bin;
                            s_above = run;
                            break;
                        }
                        run += tot[bin];
                    }
                }
            }
            __syncthreads();
            remaining -= s_above;
            prefix |= s_bin << shift;
            mask |= 255u << shift;
        }
    } else {
        prefix = 0xffffffffu;  // nothing above it, no equal candidate taken
    }
    const uint32_t kth = prefix;
    const uint32_t need_eq = k > 0 ? remaining : 0u;

    // ---- ordered compaction: each thread owns a contiguous run of positions
    const int n = hi - lo;
    const int seg = (n + SEL_NT - 1) / SEL_NT;
    const int s0 = lo + min(n, tid * seg), s1 = lo + min(n, (tid + 1) * seg);
    uint32_t n_eq = 0;
    for (int p = s0; p < s1; ++p)
        if (p >= cand_lo && p < cand_hi && keys[p - lo] == kth) ++n_eq;
    uint32_t eq_cta;
    const uint32_t eq_before = block_excl_scan<SEL_NT>(n_eq, wsum, &eq_cta);
    if (tid == 0) xch[0] = eq_cta;
    cluster.sync();
    uint32_t eq_base = 0;
    for (int r = 0; r < rank; ++r) eq_base += cluster.map_shared_rank(xch, r)[0];
    uint32_t run_eq = eq_base + eq_before, n_sel = 0;
    for (int p = s0; p < s1; ++p) {
        bool s;
        if (p < cand_lo || p >= cand_hi) {
            s = true;
        } else {
            const uint32_t key = keys[p - lo];
            s = key > kth;
            if (key == kth) s = (run_eq++ < need_eq);
        }
        n_sel += s;
    }
    uint32_t sel_cta;
    const uint32_t sel_before = block_excl_scan<SEL_NT>(n_sel, wsum, &sel_cta);
    if (tid == 0) xch[1] = sel_cta;
    cluster.sync();
    uint32_t sel_base = 0;
    for (int r = 0; r < rank; ++r) sel_base += cluster.map_shared_rank(xch, r)[1];
    uint32_t o_idx = sel_base + sel_before;
    run_eq = eq_base + eq_before;
    bool overflow = false;
    for (int p = s0; p < s1; ++p) {
        bool s;
        if (p < cand_lo || p >= cand_hi) {
            s = true;
        } else {
            const uint32_t key = keys[p - lo];
            s = key > kth;
            if (key == kth) s = (run_eq++ < need_eq);
        }
        if (s) {
            if (o_idx < (uint32_t)a.sel_cap) out[o_idx] = p;
            else overflow = true;
            ++o_idx;
        }
    }
    if (overflow) kvq_dev_flag(a.hdr, KVQ_DEV_OVERFLOW, b);
    if (rank == 0 && tid == 0) {
        const int total = a.n_sink + a.window + k;
        a.sel_count[(int64_t)b * a.n_heads + h] = min(total, a.sel_cap);
    }
    cluster.sync();  // no CTA leaves while another may still read its shared memory
}

// ================================================================ a6 sparse attention

constexpr int SA_NT = 256;
constexpr int SA_HW = SA_NT / 16;  // half-warps per CTA
constexpr int SA_BATCH = 4;        // rows in flight per half-warp
constexpr int SA_REC = 4 + D;

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
    const int64_t head_stride = (int64_t)PG * D;
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
            if (i < r_end) {
                const int t = ids[i];
                if (t >= 0 && t < T) {
                    const int32_t page = a.bt[(int64_t)b * a.max_blocks + (t >> 4)];
                    if (page >= 0 && page < a.num_blocks) {
                        const int64_t off = ((int64_t)page * a.H + g) * head_stride + (int64_t)(t & 15) * D + 8 * l16;
                        kr[j] = __ldg(reinterpret_cast<const uint4*>(a.k16 + off));
                        vr[j] = __ldg(reinterpret_cast<const uint4*>(a.v16 + off));
                        ok[j] = true;
                    } else if (l16 == 0) {
                        kvq_dev_flag(a.hdr, KVQ_DEV_BAD_PAGE, t);
                    }
                } else if (l16 == 0) {
                    kvq_dev_flag(a.hdr, KVQ_DEV_BAD_INDEX, t);
                }
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
    for (int hh = 0; hh < NH; ++hh) {
        float* pr = a.probs + ((int64_t)b * Hq + h0 + hh) * a.sel_cap;
        const float M = fin_m[hh], L = fin_l[hh];
        for (int i = tid; i < n; i += SA_NT) {
            const float sv = __ldcg(pr + i);
            pr[i] = (L > 0.0f && sv != -INFINITY) ? exp2f(sv - M) / L : 0.0f;
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
    rps = std::max(64, (rps + 63) / 64 * 64);
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
    const size_t smem = (size_t)SA_HW * NH * SA_REC * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_sparse_attn: %s", cudaGetErrorString(e));
    }
    sparse_attn_kernel<NH><<<grid, SA_NT, smem, s>>>(a);
    return kvq_launch_status("kv_sparse_attn");
}

}  // namespace

// ================================================================ ABI

extern "C" int kv_critical_score(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q,
                                 int32_t n_crit, int32_t* crit, float* scores, int64_t score_stride,
                                 void* stream) {
    kvq_clear_error();
    int st = kvq_check_layout(L, "kv_critical_score", true);
    if (st) return st;
    st = kvq_check_seqs(S, "kv_critical_score");
    if (st) return st;
    KVQ_REQUIRE(P && P->kT && P->k_absmax, KVQ_ERR_INVALID_ARG, "kv_critical_score: pool needs kT and k_absmax");
    KVQ_REQUIRE(n_crit >= 1 && n_crit <= D, KVQ_ERR_INVALID_ARG, "kv_critical_score: n_crit %d not in [1, 128]", n_crit);
    KVQ_REQUIRE(P->t_cap % 8 == 0 && P->t_cap >= S->max_len, KVQ_ERR_INVALID_ARG,
                "kv_critical_score: t_cap must be a multiple of 8 and >= max_len");
    KVQ_REQUIRE(((uintptr_t)P->kT & 15u) == 0, KVQ_ERR_INVALID_ARG, "kv_critical_score: kT must be 16-byte aligned");
    KVQ_REQUIRE(scores && ((uintptr_t)scores & 15u) == 0 && score_stride % 4 == 0 && score_stride >= S->max_len,
                KVQ_ERR_INVALID_ARG, "kv_critical_score: scores must be 16-byte aligned, stride %% 4 == 0, >= max_len");
    KVQ_REQUIRE(S->batch <= P->max_seqs, KVQ_ERR_INVALID_ARG, "kv_critical_score: batch exceeds max_seqs");
    if (S->batch == 0) return KVQ_OK;
    KVQ_REQUIRE(q != nullptr, KVQ_ERR_INVALID_ARG, "kv_critical_score: NULL q");
    CritArgs a;
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
    const int tiles = std::max(1, (S->max_len + CS_TILE - 1) / CS_TILE);
    crit_score_kernel<<<dim3(tiles, L->n_q_heads, S->batch), CS_NT, 0, kvq_stream(stream)>>>(a);
    return kvq_launch_status("kv_critical_score");
}

extern "C" size_t kv_topk_select_ws(void) { return sizeof(KvqWsHeader); }

extern "C" int kv_topk_select(const kvq_seqs* S, int32_t n_heads, const float* scores, int64_t score_stride,
                              int32_t k_fixed, double ratio, int32_t n_sink, int32_t window, int32_t* sel,
                              int32_t sel_cap, int32_t* sel_count, void* ws, size_t ws_bytes, void* stream) {
    kvq_clear_error();
    int st = kvq_check_seqs(S, "kv_topk_select");
    if (st) return st;
    st = kvq_check_ws(ws, ws_bytes, kv_topk_select_ws(), "kv_topk_select");
    if (st) return st;
    KVQ_REQUIRE(n_heads > 0, KVQ_ERR_INVALID_ARG, "kv_topk_select: n_heads");
    KVQ_REQUIRE(n_sink >= 0 && window >= 0 && sel_cap > 0, KVQ_ERR_INVALID_ARG, "kv_topk_select: sizes");
    KVQ_REQUIRE(k_fixed >= 0 || (ratio >= 0.0 && ratio <= 1.0), KVQ_ERR_INVALID_ARG, "kv_topk_select: ratio");
    KVQ_REQUIRE(scores && sel && sel_count && score_stride >= S->max_len, KVQ_ERR_INVALID_ARG,
                "kv_topk_select: NULL buffer or score_stride < max_len");
    const int chunk = (S->max_len + SEL_CL - 1) / SEL_CL;
    KVQ_REQUIRE(chunk <= SEL_MAX_CHUNK, KVQ_ERR_UNSUPPORTED, "kv_topk_select: max_len %d above %d", S->max_len,
                SEL_CL * SEL_MAX_CHUNK);
    if (S->batch == 0) return KVQ_OK;
    SelArgs a;
    a.scores = scores;
    a.score_stride = score_stride;
    a.seq_lens = S->seq_lens;
    a.max_len = S->max_len;
    a.n_heads = n_heads;
    a.k_fixed = k_fixed;
    a.ratio = ratio;
    a.n_sink = n_sink;
    a.window = window;
    a.sel = sel;
    a.sel_cap = sel_cap;
    a.sel_count = sel_count;
    a.hdr = static_cast<KvqWsHeader*>(ws);
    const size_t smem = (size_t)std::max(chunk, 1) * sizeof(uint32_t);
    static int configured = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured != dev) {
        cudaError_t e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SEL_MAX_CHUNK * (int)sizeof(uint32_t));
        if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_topk_select: %s", cudaGetErrorString(e));
        configured = dev;
    }
    topk_select_kernel<<<dim3(SEL_CL, n_heads, S->batch), SEL_NT, smem, kvq_stream(stream)>>>(a);
    return kvq_launch_status("kv_topk_select");
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
