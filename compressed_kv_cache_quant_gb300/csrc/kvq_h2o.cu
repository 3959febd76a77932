// a7 kv_h2o_accumulate [KVSurvey §三.2, §三.1] and a8 kv_dense_pref_score
// [TailorKV §2.1].
#include <algorithm>

#include "kvq_internal.cuh"

namespace {

constexpr int D = KVQ_HEAD_DIM;
constexpr int PG = KVQ_BLOCK_TOKENS;

// ================================================================ a7 H2O accumulate / evict / admit

constexpr int HA_NT = 1024;

constexpr int HA_U = 4;        // list entries per thread and pass step (their loads in flight together)

struct H2OArgs {
    const float* probs;      // [B][H_q][cap]
    int32_t* retained;
    int32_t* count;
    float* cum;
    int32_t cap;
    int32_t budget, n_sink, window;
    const int32_t* new_pos;
    int32_t* n_evicted;
    const int32_t* seq_lens;
    int32_t H, GQ;
    KvqWsHeader* hdr;
};

// Eviction order: lowest cumulative score first, then lowest position.
__device__ __forceinline__ unsigned long long evict_key(float cum, int32_t pos) {
    return ((unsigned long long)kvq_float_key(cum) << 32) | (uint32_t)pos;
}

__device__ __forceinline__ uint32_t block_sum_u32(uint32_t v, uint32_t* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    uint32_t s = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
    return s;
}

// Evicts the `excess` (> 1) unprotected entries of lowest (cum, position) key from ret/cum[0, n)
// (all of them when there are no more), keeping the order of the others; returns the new length.
// Called by all NTH threads of a CTA.
template <int NTH>
__device__ int h2o_evict_many(int32_t* ret, float* cum, int n, int excess, int n_sink, int window, int next_len) {
    __shared__ uint32_t red[NTH / 32];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_bin, s_below;
    __shared__ uint32_t wsum[NTH / 32];
    const int tid = threadIdx.x;
    auto is_protected = [&](int32_t pos) { return pos < n_sink || pos >= next_len - window; };
    uint32_t n_un = 0;
    for (int i = tid; i < n; i += NTH) n_un += !is_protected(ret[i]);
    const uint32_t U = block_sum_u32(n_un, red);
    unsigned long long thr;
    if (U <= (uint32_t)excess) {
        thr = ~0ull;  // every unprotected token goes
    } else {
        // radix select of the excess-th smallest 64-bit key among unprotected tokens
        unsigned long long prefix = 0ull, mask = 0ull;
        uint32_t remaining = (uint32_t)excess;
        for (int pass = 0; pass < 8; ++pass) {
            const int shift = 56 - 8 * pass;
            for (int i = tid; i < 256; i += NTH) hist[i] = 0u;
            __syncthreads();
            for (int i = tid; i < n; i += NTH) {
                const int32_t pos = ret[i];
                if (is_protected(pos)) continue;
                const unsigned long long k = evict_key(cum[i], pos);
                if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255ull], 1u);
            }
            __syncthreads();
            if (tid < 32) {
                // lane l owns bins [8l, 8l + 7]; lane 0 the smallest
                uint32_t ls = 0;
                for (int j = 0; j < 8; ++j) ls += hist[8 * tid + j];
                uint32_t incl = ls;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (tid >= o) incl += y;
                }
                const uint32_t ballot = __ballot_sync(0xffffffffu, incl >= remaining);
                const int l = __ffs(ballot) - 1;
                if (tid == l) {
                    uint32_t run = incl - ls;
                    for (int j = 0; j < 8; ++j) {
                        const int bin = 8 * tid + j;
                        if (run + hist[bin] >= remaining) {
                            s_bin = (uint32_t)bin;
                            s_below = run;
                            break;
                        }
                        run += hist[bin];
                    }
                }
            }
            __syncthreads();
            remaining -= s_below;
            prefix |= (unsigned long long)s_bin << shift;
            mask |= 255ull << shift;
            __syncthreads();
        }
        thr = prefix;
    }
    // order-preserving in-place compaction of the kept entries
    uint32_t out_base = 0;
    for (int t0 = 0; t0 < n; t0 += NTH) {
        const int i = t0 + tid;
        int32_t pos = 0;
        float cv = 0.0f;
        uint32_t keep = 0;
        if (i < n) {
            pos = ret[i];
            cv = cum[i];
            keep = is_protected(pos) || evict_key(cv, pos) > thr;
        }
        uint32_t tile_total;
        // exclusive scan of `keep` over the CTA
        const int lane = tid & 31, warp = tid >> 5;
        uint32_t x = keep;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        __syncthreads();
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            uint32_t w = lane < NTH / 32 ? wsum[lane] : 0u;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        tile_total = wsum[NTH / 32 - 1];
        const uint32_t before = x - keep + (warp > 0 ? wsum[warp - 1] : 0u);
        if (keep) {
            ret[out_base + before] = pos;
            cum[out_base + before] = cv;
        }
        out_base += tile_total;
        __syncthreads();
    }
    return (int)out_base;
}

__global__ void __launch_bounds__(HA_NT) h2o_kernel(H2OArgs a) {
    __shared__ unsigned long long redk[HA_NT / 32];
    const int g = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    kvq_pdl_begin();
    const int Hq = a.H * a.GQ;
    const int64_t base = ((int64_t)b * a.H + g) * a.cap;
    int32_t* ret = a.retained + base;
    float* cum = a.cum + base;
    int n = a.count[(int64_t)b * a.H + g];
    if (n < 0 || n > a.cap) {
        if (tid == 0) kvq_dev_flag(a.hdr, KVQ_DEV_OVERFLOW, b);
        n = max(0, min(n, a.cap));
    }
    const int T = a.seq_lens[b];
    const int next_len = T + 1;
    const int newp = a.new_pos ? a.new_pos[b] : -1;
    const int target = newp >= 0 ? a.budget - 1 : a.budget;
    const int excess = n - target;
    int evicted = 0;
    auto is_protected = [&](int32_t pos) { return pos < a.n_sink || pos >= next_len - a.window; };
    // 1. cum += p_0 + p_1 + ... (the group's heads in ascending order, fp32).  When exactly one
    //    token goes, the same pass finds it: the lowest (cum, position) key among the unprotected
    //    entries, with its index.
    const float* const pr = a.probs + ((int64_t)b * Hq + g * a.GQ) * a.cap;
    unsigned long long best = ~0ull;
    int best_i = -1;
    for (int i0 = tid; i0 < n; i0 += HA_U * HA_NT) {
        float cv[HA_U], inc[HA_U];
        int32_t pv[HA_U];
#pragma unroll
        for (int u = 0; u < HA_U; ++u) {
            const int i = i0 + u * HA_NT;
            cv[u] = i < n ? cum[i] : 0.0f;
            pv[u] = i < n ? ret[i] : 0;
            inc[u] = 0.0f;
        }
        for (int hh = 0; hh < a.GQ; ++hh) {
            const float* const ph = pr + (int64_t)hh * a.cap;
            float sv[HA_U];
#pragma unroll
            for (int u = 0; u < HA_U; ++u) sv[u] = i0 + u * HA_NT < n ? ph[i0 + u * HA_NT] : 0.0f;
#pragma unroll
            for (int u = 0; u < HA_U; ++u) inc[u] = hh == 0 ? sv[u] : inc[u] + sv[u];
        }
#pragma unroll
        for (int u = 0; u < HA_U; ++u) {
            const int i = i0 + u * HA_NT;
            if (i < n) {
                const float c = cv[u] + inc[u];
                cum[i] = c;
                if (excess == 1 && !is_protected(pv[u])) {
                    const unsigned long long k = evict_key(c, pv[u]);
                    if (k < best) {
                        best = k;
                        best_i = i;
                    }
                }
            }
        }
    }
    __syncthreads();
    // 2. evict unprotected tokens, lowest (cum, position) first
    if (excess == 1) {
        // the block's minimum key and its index (positions are unique: one entry carries it)
        __shared__ int redi[HA_NT / 32];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long k2 = __shfl_xor_sync(0xffffffffu, best, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, best_i, o);
            if (k2 < best) {
                best = k2;
                best_i = i2;
            }
        }
        if ((tid & 31) == 0) {
            redk[tid >> 5] = best;
            redi[tid >> 5] = best_i;
        }
        __syncthreads();
        if (tid == 0) {
            unsigned long long kmin = redk[0];
            int imin = redi[0];
            for (int w = 1; w < HA_NT / 32; ++w)
                if (redk[w] < kmin) {
                    kmin = redk[w];
                    imin = redi[w];
                }
            if (kmin != ~0ull) {
                ret[imin] = ret[n - 1];
                cum[imin] = cum[n - 1];
                n -= 1;
                evicted = 1;
            }
        }
    } else if (excess > 1) {
        const int kept = h2o_evict_many<HA_NT>(ret, cum, n, excess, a.n_sink, a.window, next_len);
        evicted = n - kept;
        n = kept;
    }
    // 3. admit the next token with score 0
    if (tid == 0) {
        if (newp >= 0) {
            if (n < a.cap) {
                ret[n] = newp;
                cum[n] = 0.0f;
                ++n;
            } else {
                kvq_dev_flag(a.hdr, KVQ_DEV_OVERFLOW, b);
            }
        }
        a.count[(int64_t)b * a.H + g] = n;
        if (a.n_evicted) a.n_evicted[(int64_t)b * a.H + g] = evicted;
    }
}

// ================================================================ a8 dense-preference score
//
// Two launches.  dp_scores_kernel, per (128-token tile, kv head, sequence): the scores of all the
// kv head's R = GQ n_q query rows against the tile's keys as m16n8k16 tensor-core products (fp16
// inputs, exact products, fp32 sums; channels permuted inside each k-step identically in both
// operands so that every lane reads whole 8-byte runs), scaled to the log2 domain and written to
// the workspace score matrix [B][H_q][n_q][ld]: K is read once per kv head, not once per query.
// dp_row_kernel, per row (query i of q head h of sequence b) over its causal prefix L = T - n_q +
// i + 1: max and sum of exp2 (one online pass), the k-th largest score by a four-pass 8-bit radix
// select on order-preserving keys, the top-k mass; the last row of (b, h) forms P.  A row of up to
// DP_SMEM_T scores is copied to shared memory first; a longer row is read from the workspace in
// every pass (no length limit).

constexpr int DP_NT = 256;
constexpr int DP_SMEM_T = 40960;         // rows up to this length are reduced in shared memory
constexpr int DPS_NW = 8;                // warps of the scores kernel: one 16-token page each
constexpr int DPS_TILE = DPS_NW * PG;    // tokens per scores CTA
constexpr int DPS_QLD = D + 16;          // padded query row in shared memory (halves, 288 bytes)
constexpr int DP_MAX_ROWS = 512;         // GQ n_q query rows of one kv head

struct DPArgs {
    const uint16_t* k16;
    int64_t num_blocks;
    const int32_t* bt;
    const int32_t* seq_lens;
    int32_t max_blocks, max_len;
    int32_t H, GQ;
    const uint16_t* q;
    int32_t n_q, topk;
    float* P;
    float* S;           // [B][H_q][n_q][ld] log2-domain scores
    int64_t ld;
    int32_t smem_cap;   // scores the row kernel's shared memory holds (0: every row read from S)
    float* rows;        // [B][H_q][n_q] per-query top-k mass
    int32_t* counters;  // [B][H_q]
    KvqWsHeader* hdr;
};

__device__ __forceinline__ void dp_mma(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(32 * DPS_NW) dp_scores_kernel(DPArgs a) {
    extern __shared__ __align__(16) uint16_t qsm[];  // [R16][DPS_QLD]
    const int tile = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g8 = lane >> 2, q4 = lane & 3;
    const int R = a.GQ * a.n_q, R16 = (R + 15) & ~15;
    const int Hq = a.H * a.GQ;
    const int T = a.seq_lens[b];
    if (T > a.max_len || T < 0) {
        if (tid == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
        return;
    }
    const int t_base = tile * DPS_TILE;
    if (t_base >= T) return;
    // the kv head's query rows (row j n_q + i: query i of q head g GQ + j), zero rows up to R16
    const uint16_t* qsrc = a.q + ((int64_t)b * Hq + g * a.GQ) * a.n_q * D;
    for (int e = tid; e < R16 * (D / 8); e += 32 * DPS_NW) {
        const int r = e / (D / 8), c8 = e % (D / 8);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < R) v = __ldg(reinterpret_cast<const uint4*>(qsrc + (int64_t)r * D + 8 * c8));
        *reinterpret_cast<uint4*>(qsm + r * DPS_QLD + 8 * c8) = v;
    }
    __syncthreads();
    const int t0 = t_base + warp * PG;  // this warp's page
    if (t0 >= T) return;                // (no block barrier below)
    int32_t page = a.bt[(int64_t)b * a.max_blocks + t0 / PG];
    if (page < 0 || page >= a.num_blocks) {
        if (lane == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_PAGE, t0);
        return;
    }
    // B fragments of the page's tokens g8 (n-tile 0) and g8 + 8 (n-tile 1): k slot 2 q4 + e of k-step
    // s is channel 16 s + 4 q4 + e, slot 8 + 2 q4 + e is channel 16 s + 4 q4 + 2 + e (the A operand
    // below uses the same map, so the sums are the dot products over all 128 channels)
    uint32_t kb[2][8][2];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
        const int tok = g8 + 8 * n;
        const bool valid = t0 + tok < T;
        const uint16_t* kr = a.k16 + (((int64_t)page * a.H + g) * PG + tok) * D + 4 * q4;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint2 w = valid ? __ldg(reinterpret_cast<const uint2*>(kr + 16 * s)) : make_uint2(0u, 0u);
            kb[n][s][0] = w.x;
            kb[n][s][1] = w.y;
        }
    }
    float* srow = a.S + ((int64_t)b * Hq + g * a.GQ) * a.n_q * a.ld;  // row r at srow + r ld
    for (int mt = 0; mt < R16 / 16; ++mt) {
        float d[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) d[n][0] = d[n][1] = d[n][2] = d[n][3] = 0.0f;
        const uint16_t* q0 = qsm + (16 * mt + g8) * DPS_QLD + 4 * q4;
        const uint16_t* q1 = q0 + 8 * DPS_QLD;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint2 x0 = *reinterpret_cast<const uint2*>(q0 + 16 * s);
            const uint2 x1 = *reinterpret_cast<const uint2*>(q1 + 16 * s);
#pragma unroll
            for (int n = 0; n < 2; ++n) dp_mma(d[n], x0.x, x1.x, x0.y, x1.y, kb[n][s][0], kb[n][s][1]);
        }
        // d[n][0..1]: row 16 mt + g8, tokens t0 + 8 n + 2 q4 + {0, 1}; d[n][2..3]: row 16 mt + g8 + 8
        const int r0 = 16 * mt + g8, r1 = r0 + 8;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const int tt = t0 + 8 * n + 2 * q4;
            if (r0 < R)
                *reinterpret_cast<float2*>(srow + (int64_t)r0 * a.ld + tt) =
                    make_float2(d[n][0] * KVQ_SCORE_LOG2_SCALE, d[n][1] * KVQ_SCORE_LOG2_SCALE);
            if (r1 < R)
                *reinterpret_cast<float2*>(srow + (int64_t)r1 * a.ld + tt) =
                    make_float2(d[n][2] * KVQ_SCORE_LOG2_SCALE, d[n][3] * KVQ_SCORE_LOG2_SCALE);
        }
    }
}

__device__ __forceinline__ float block_reduce_max(float v, float* red) {
    v = kvq_warp_max(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = fmaxf(r, red[w]);
    return r;
}

__device__ __forceinline__ float block_reduce_sum(float v, float* red) {
    v = kvq_warp_sum(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r += red[w];
    return r;
}

// Adds 1 to bin `bin` of the histogram h (bin >= nb: nothing), equal bins of the warp's lanes
// combined into one shared-memory atomic.  Called by all 32 lanes.
__device__ __forceinline__ void dp_hist_add(uint32_t* h, uint32_t bin, uint32_t nb) {
    const uint32_t peers = __match_any_sync(0xffffffffu, bin);
    if (bin < nb && (threadIdx.x & 31) == (unsigned)(__ffs(peers) - 1)) atomicAdd(&h[bin], (uint32_t)__popc(peers));
}

// The float whose order-preserving key is k (kvq_float_key; -0 reads as +0)
__device__ __forceinline__ float dp_key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

constexpr int DP_H1 = 2048;       // first digit: the keys' top 11 bits
constexpr int DP_CAND = 6144;     // scores of the k-th key's first-digit bin kept in shared memory

// Over nb bins (a multiple of DP_NT: nb / DP_NT consecutive bins per thread, thread 0 the highest),
// finds from the top the bin holding the `remaining`-th largest element: *bin, and *above = the
// count in the higher bins.  Called by the whole CTA; ends with a barrier.
__device__ __forceinline__ void dp_find_bin(const uint32_t* h, int nb, uint32_t remaining, uint32_t* bin,
                                            uint32_t* above, uint32_t* wsum) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = nb / DP_NT;                 // bins per thread, thread 0 the highest
    const int top = nb - per * tid;             // this thread's bins: top - per .. top - 1
    uint32_t mine = 0;
    for (int j = 0; j < per; ++j) mine += h[top - 1 - j];
    uint32_t x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    uint32_t before = 0;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    uint32_t run = before + x - mine;           // the count above this thread's bins
    if (run < remaining && run + mine >= remaining) {
        for (int j = 0; j < per; ++j) {
            const uint32_t c = h[top - 1 - j];
            if (run + c >= remaining) {
                *bin = (uint32_t)(top - 1 - j);
                *above = run;
                break;
            }
            run += c;
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(DP_NT) dp_row_kernel(DPArgs a) {
    extern __shared__ __align__(16) float sc[];  // the row, when it has at most a.smem_cap scores
    constexpr int NWR = DP_NT / 32;
    __shared__ float redf[NWR];
    __shared__ uint32_t wsum[NWR];
    __shared__ uint32_t hist[DP_H1];             // digit histograms (2048 bins, then 256)
    __shared__ float cand[DP_CAND];              // the first-digit bin's scores
    __shared__ uint32_t s_bin, s_above, n_cand;
    __shared__ int is_last;
    const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hq = a.H * a.GQ;
    const int T = a.seq_lens[b];
    const int L = T - a.n_q + i + 1;  // keys seen by query i
    float r_i = 0.0f;
    if (T > a.max_len || L <= 0) {
        if (tid == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
    } else {
        // the row: ld >= L rounded up to 128 floats, 512-byte aligned, so whole float4 groups may be
        // read past L (their extra lanes are masked)
        const float* row = a.S + (((int64_t)b * Hq + h) * a.n_q + i) * a.ld;
        const int L4 = (L + 3) >> 2;
        const bool in_smem = L <= a.smem_cap;
        if (in_smem)
            for (int t = tid; t < L4; t += DP_NT)
                reinterpret_cast<float4*>(sc)[t] = __ldcg(reinterpret_cast<const float4*>(row) + t);
        for (int j = tid; j < DP_H1; j += DP_NT) hist[j] = 0u;
        if (tid == 0) n_cand = 0u;
        __syncthreads();
        const float4* src = reinterpret_cast<const float4*>(in_smem ? sc : row);
        const int kk = min(a.topk, L);
        // pass 1: max and sum of exp2 (a running sum rescaled when the running max grows) and the
        // histogram of the keys' top 11 bits; the loops walk warp-uniform blocks of 32 float4s
        float mx = -INFINITY, z = 0.0f;
        for (int t0 = 32 * warp; t0 < L4; t0 += DP_NT) {
            const int t4 = t0 + lane;
            float v[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (t4 < L4) {
                const float4 x = src[t4];
                v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint32_t bin = DP_H1;
                if (4 * t4 + e < L) {
                    if (v[e] > mx) {
                        z = fmaf(z, exp2f(mx - v[e]), 1.0f);
                        mx = v[e];
                    } else {
                        z += exp2f(v[e] - mx);
                    }
                    bin = kvq_float_key(v[e]) >> 21;
                }
                dp_hist_add(hist, bin, DP_H1);
            }
        }
        const float M = block_reduce_max(mx, redf);
        z = block_reduce_sum(mx == -INFINITY ? 0.0f : z * exp2f(mx - M), redf);  // (synchronizes)
        dp_find_bin(hist, DP_H1, (uint32_t)kk, &s_bin, &s_above, wsum);
        const uint32_t b1 = s_bin;
        const uint32_t rem1 = (uint32_t)kk - s_above;  // still to take from bin b1
        // pass 2: the mass of the bins above b1; bin b1's scores into the candidate buffer
        float top = 0.0f;
        for (int t0 = 32 * warp; t0 < L4; t0 += DP_NT) {
            const int t4 = t0 + lane;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t4 < L4) x = src[t4];
            const float v[4] = {x.x, x.y, x.z, x.w};
            bool cf[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool ok = 4 * t4 + e < L;
                const uint32_t bin = ok ? kvq_float_key(v[e]) >> 21 : 0u;
                if (ok && bin > b1) top += exp2f(v[e] - M);
                cf[e] = ok && bin == b1;
            }
            // candidates are rare (one bin of 2048): one vote per group of four, the slots only
            // when a lane of the warp has one
            if (__any_sync(0xffffffffu, cf[0] || cf[1] || cf[2] || cf[3])) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t bal = __ballot_sync(0xffffffffu, cf[e]);
                    uint32_t base = 0;
                    if (lane == 0 && bal != 0u) base = atomicAdd(&n_cand, (uint32_t)__popc(bal));
                    base = __shfl_sync(0xffffffffu, base, 0) + (uint32_t)__popc(bal & ((1u << lane) - 1u));
                    if (cf[e] && base < (uint32_t)DP_CAND) cand[base] = v[e];
                }
            }
        }
        for (int j = tid; j < DP_H1; j += DP_NT) hist[j] = 0u;
        __syncthreads();
        // the low 21 bits of the k-th key among bin b1's scores: digits of 8, 8 and 5 bits over the
        // candidate buffer, or, if it overflowed (more than DP_CAND equal top bits), over the row
        const uint32_t nc = n_cand;
        const bool in_buf = nc <= (uint32_t)DP_CAND;
        uint32_t prefix = b1 << 21, mask = 0xffe00000u, remaining = rem1;
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = pass == 0 ? 13 : pass == 1 ? 5 : 0;
            const uint32_t dm = pass == 2 ? 31u : 255u;
            if (in_buf) {
                for (int j0 = 32 * warp; j0 < (int)nc; j0 += DP_NT) {
                    const int j = j0 + lane;
                    uint32_t bin = 256u;
                    if (j < (int)nc) {
                        const uint32_t key = kvq_float_key(cand[j]);
                        if ((key & mask) == prefix) bin = (key >> shift) & dm;
                    }
                    dp_hist_add(hist, bin, 256u);
                }
            } else {
                for (int t0 = 32 * warp; t0 < L4; t0 += DP_NT) {
                    const int t4 = t0 + lane;
                    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (t4 < L4) x = src[t4];
                    const float v[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint32_t bin = 256u;
                        if (4 * t4 + e < L) {
                            const uint32_t key = kvq_float_key(v[e]);
                            if ((key & mask) == prefix) bin = (key >> shift) & dm;
                        }
                        dp_hist_add(hist, bin, 256u);
                    }
                }
            }
            __syncthreads();
            dp_find_bin(hist, 256, remaining, &s_bin, &s_above, wsum);
            remaining -= s_above;
            prefix |= s_bin << shift;
            mask |= dm << shift;
            for (int j = tid; j < 256; j += DP_NT) hist[j] = 0u;
            __syncthreads();
        }
        // prefix is the k-th key: bin b1's scores above it join the mass, and the k-th value fills
        // the slots left (ties at the k-th key)
        float top2 = 0.0f;
        uint32_t n_gt2 = 0;
        if (in_buf) {
            for (int j = tid; j < (int)nc; j += DP_NT) {
                const float v = cand[j];
                if (kvq_float_key(v) > prefix) {
                    top2 += exp2f(v - M);
                    ++n_gt2;
                }
            }
        } else {
            for (int t4 = tid; t4 < L4; t4 += DP_NT) {
                const float4 x = src[t4];
                const float v[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (4 * t4 + e >= L) break;
                    const uint32_t key = kvq_float_key(v[e]);
                    if ((key >> 21) == b1 && key > prefix) {
                        top2 += exp2f(v[e] - M);
                        ++n_gt2;
                    }
                }
            }
        }
        top = block_reduce_sum(top + top2, redf);
        n_gt2 = (uint32_t)block_reduce_sum((float)n_gt2, redf);
        top += (float)(rem1 - n_gt2) * exp2f(dp_key_float(prefix) - M);
        r_i = top / z;
    }
    // per-query mass -> workspace; the last CTA of (b, h) forms P = n_q - sum_i r_i
    if (tid == 0) a.rows[((int64_t)b * Hq + h) * a.n_q + i] = r_i;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(&a.counters[(int64_t)b * Hq + h], 1);
        is_last = (prev == a.n_q - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    if (tid == 0) {
        double s = 0.0;
        for (int j = 0; j < a.n_q; ++j) s += (double)__ldcg(a.rows + ((int64_t)b * Hq + h) * a.n_q + j);
        a.P[(int64_t)b * Hq + h] = (float)((double)a.n_q - s);
        a.counters[(int64_t)b * Hq + h] = 0;
    }
}

int64_t dp_ld(const kvq_seqs* S) {
    return ((int64_t)std::max(S->max_len, 1) + DPS_TILE - 1) / DPS_TILE * DPS_TILE;
}

size_t dp_ws_layout(const kvq_layout* L, const kvq_seqs* S, int32_t n_q, size_t* off_rows, size_t* off_cnt,
                    size_t* off_s) {
    const size_t rows = (size_t)std::max(S->batch, 1) * L->n_q_heads * (size_t)std::max(n_q, 1);
    *off_rows = sizeof(KvqWsHeader);
    *off_cnt = kvq_round_up(*off_rows + rows * sizeof(float), 256);
    *off_s = kvq_round_up(*off_cnt + (size_t)std::max(S->batch, 1) * L->n_q_heads * sizeof(int32_t), 256);
    return kvq_round_up(*off_s + rows * (size_t)dp_ld(S) * sizeof(float), 256);
}

}  // namespace

// ================================================================ ABI

extern "C" size_t kv_h2o_accumulate_ws(void) { return sizeof(KvqWsHeader); }

extern "C" int kv_h2o_accumulate(const kvq_layout* L, const kvq_seqs* S, const float* probs, int32_t* retained,
                                 int32_t* retained_count, float* cum, int32_t cap, int32_t budget, int32_t n_sink,
                                 int32_t window, const int32_t* new_pos, int32_t* n_evicted, void* ws,
                                 size_t ws_bytes, void* stream) {
    kvq_clear_error();
    int st = kvq_check_layout(L, "kv_h2o_accumulate", true);
    if (st) return st;
    st = kvq_check_seqs(S, "kv_h2o_accumulate");
    if (st) return st;
    st = kvq_check_ws(ws, ws_bytes, kv_h2o_accumulate_ws(), "kv_h2o_accumulate");
    if (st) return st;
    KVQ_REQUIRE(probs && retained && retained_count && cum, KVQ_ERR_INVALID_ARG, "kv_h2o_accumulate: NULL buffer");
    KVQ_REQUIRE(cap > 0 && budget >= 1 && budget <= cap && n_sink >= 0 && window >= 0, KVQ_ERR_INVALID_ARG,
                "kv_h2o_accumulate: need 1 <= budget <= cap, n_sink >= 0, window >= 0");
    if (S->batch == 0) return KVQ_OK;
    H2OArgs a{};
    a.probs = probs;
    a.retained = retained;
    a.count = retained_count;
    a.cum = cum;
    a.cap = cap;
    a.budget = budget;
    a.n_sink = n_sink;
    a.window = window;
    a.new_pos = new_pos;
    a.n_evicted = n_evicted;
    a.seq_lens = S->seq_lens;
    a.H = L->n_kv_heads;
    a.GQ = L->n_q_heads / L->n_kv_heads;
    a.hdr = static_cast<KvqWsHeader*>(ws);
    const cudaError_t e = kvq_launch_pdl(h2o_kernel, dim3(L->n_kv_heads, S->batch), dim3(HA_NT), 0, kvq_stream(stream), a);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_h2o_accumulate launch: %s", cudaGetErrorString(e));
    return kvq_launch_status("kv_h2o_accumulate");
}

extern "C" size_t kv_dense_pref_score_ws(const kvq_layout* L, const kvq_seqs* S, int32_t n_q) {
    if (kvq_check_layout(L, "kv_dense_pref_score_ws", true) || kvq_check_seqs_sizes(S, "kv_dense_pref_score_ws")) return 0;
    size_t a, c, s;
    return dp_ws_layout(L, S, n_q, &a, &c, &s);
}

extern "C" int kv_dense_pref_score(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q_recent,
                                   int32_t n_q, int32_t topk, float* Pout, void* ws, size_t ws_bytes, void* stream) {
    kvq_clear_error();
    const char* fn = "kv_dense_pref_score";
    int st = kvq_check_layout(L, fn, true);
    if (st) return st;
    st = kvq_check_seqs(S, fn);
    if (st) return st;
    KVQ_REQUIRE(P && P->k16, KVQ_ERR_INVALID_ARG, "%s: pool needs k16", fn);
    KVQ_REQUIRE(((uintptr_t)P->k16 & 15u) == 0 && ((uintptr_t)q_recent & 15u) == 0, KVQ_ERR_INVALID_ARG,
                "%s: k16 and q_recent must be 16-byte aligned", fn);
    KVQ_REQUIRE(n_q >= 1 && n_q <= S->max_len && topk >= 1, KVQ_ERR_INVALID_ARG,
                "%s: need 1 <= n_q <= max_len and topk >= 1", fn);
    const int gq = L->n_q_heads / L->n_kv_heads;
    KVQ_REQUIRE((int64_t)gq * n_q <= DP_MAX_ROWS, KVQ_ERR_UNSUPPORTED,
                "%s: (q heads per kv head) x n_q = %d above %d", fn, gq * n_q, DP_MAX_ROWS);
    size_t off_rows, off_cnt, off_s;
    const size_t need = dp_ws_layout(L, S, n_q, &off_rows, &off_cnt, &off_s);
    st = kvq_check_ws(ws, ws_bytes, need, fn);
    if (st) return st;
    if (S->batch == 0) return KVQ_OK;
    KVQ_REQUIRE(q_recent && Pout && S->block_table, KVQ_ERR_INVALID_ARG, "%s: NULL buffer", fn);
    DPArgs a;
    a.k16 = P->k16;
    a.num_blocks = P->num_blocks;
    a.bt = S->block_table;
    a.seq_lens = S->seq_lens;
    a.max_blocks = S->max_blocks;
    a.max_len = S->max_len;
    a.H = L->n_kv_heads;
    a.GQ = gq;
    a.q = q_recent;
    a.n_q = n_q;
    a.topk = topk;
    a.P = Pout;
    a.S = reinterpret_cast<float*>(static_cast<char*>(ws) + off_s);
    a.ld = dp_ld(S);
    a.rows = reinterpret_cast<float*>(static_cast<char*>(ws) + off_rows);
    a.counters = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + off_cnt);
    a.hdr = static_cast<KvqWsHeader*>(ws);
    cudaStream_t s = kvq_stream(stream);
    const int r16 = (gq * n_q + 15) & ~15;
    const int smem_q = r16 * DPS_QLD * (int)sizeof(uint16_t);
    st = kvq_prepare_kernel((const void*)dp_scores_kernel, smem_q);
    if (st) return st;
    const unsigned tiles = (unsigned)((std::max(S->max_len, 1) + DPS_TILE - 1) / DPS_TILE);
    dp_scores_kernel<<<dim3(tiles, L->n_kv_heads, S->batch), 32 * DPS_NW, smem_q, s>>>(a);
    st = kvq_launch_status(fn);
    if (st) return st;
    // rows up to DP_SMEM_T scores are reduced in shared memory; when the longest row is longer, no
    // shared memory is reserved (every row is read from the workspace) so that many rows share an SM
    a.smem_cap = S->max_len <= DP_SMEM_T ? (std::max(S->max_len, 1) + 3) / 4 * 4 : 0;
    const int smem_row = a.smem_cap * (int)sizeof(float);
    st = kvq_prepare_kernel((const void*)dp_row_kernel, smem_row);
    if (st) return st;
    dp_row_kernel<<<dim3(n_q, L->n_q_heads, S->batch), DP_NT, smem_row, s>>>(a);
    return kvq_launch_status(fn);
}
