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

// NHS query heads per score row: 1 = one row per q head (a4); NHS = GQ = one row per kv head,
// its group's per-head scores summed (f1, the selection shared by a GQA group).
template <int NHS>
__global__ void __launch_bounds__(CS_NT, NHS <= 2 ? CS_MINB : 2) crit_score_kernel(CritArgs a) {
    __shared__ float sc[D];
    __shared__ float qs[NHS][D];
    __shared__ uint16_t knew[D];
    __shared__ int32_t clist[D];
    __shared__ uint32_t lhist[CS_H1];
    const int tid = threadIdx.x;
    const int Hq = a.H * a.GQ;
    const int R = NHS == 1 ? Hq : a.H;  // score rows per sequence
    const int i_begin = (int)(((int64_t)a.n_items * blockIdx.x) / gridDim.x);
    const int i_end = (int)(((int64_t)a.n_items * (blockIdx.x + 1)) / gridDim.x);
    int cur = -1;  // (sequence, row) whose channels and histogram are held
    int T = 0, p_new = -1, cand_lo = 0, cand_hi = 0;
    if (a.hist != nullptr)
        for (int i = tid; i < CS_H1; i += CS_NT) lhist[i] = 0u;
    for (int item = i_begin; item < i_end; ++item) {
        const int rowi = item / a.tiles, tile = item % a.tiles;
        const int b = rowi / R, r = rowi % R;
        const int g = NHS == 1 ? r / a.GQ : r;
        const int h = NHS == 1 ? r : g * a.GQ;  // the row's first q head
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
                float am = a.absmax[kvrow * D + tid];
                if (p_new >= 0) {
                    const uint16_t kn = a.k_new[kvrow * D + tid];
                    knew[tid] = kn;
                    am = fmaxf(am, fabsf(kvq_h2f(kn)));
                }
                // sum over the row's heads of |q_c| (fp32, ascending head), times max|K_c|; for one
                // head both factors are fp16 values, so the fp32 product is exact
                float qa = 0.0f;
#pragma unroll
                for (int j = 0; j < NHS; ++j) {
                    const float qv = kvq_h2f(a.q[((int64_t)b * Hq + h + j) * D + tid]);
                    qs[j][tid] = qv;
                    qa = j == 0 ? fabsf(qv) : __fadd_rn(qa, fabsf(qv));
                }
                sc[tid] = __fmul_rn(qa, am);
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
        float accs[NHS][CS_TOK];
#pragma unroll
        for (int j = 0; j < NHS; ++j)
#pragma unroll
            for (int i = 0; i < CS_TOK; ++i) accs[j][i] = 0.0f;
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
                for (int hh = 0; hh < NHS; ++hh) {
                    const float qc = qs[hh][c];
#pragma unroll
                    for (int i = 0; i < CS_TOK; ++i) accs[hh][i] = fmaf(qc, k[i], accs[hh][i]);
                }
            }
        }
        // the row's score: its heads' scores summed in ascending head order (fp32)
        float acc[CS_TOK];
#pragma unroll
        for (int i = 0; i < CS_TOK; ++i) {
            acc[i] = accs[0][i];
#pragma unroll
            for (int hh = 1; hh < NHS; ++hh) acc[i] = __fadd_rn(acc[i], accs[hh][i]);
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

// Tensor-core form: a warp takes 16 listed rows at a time (its own tiles, staged sa_stages(NH) - 1
// tiles ahead with cp.async).  Scores S^T (heads x 16 rows) = Q K^T with m16n8k16 products: A =
// the q rows (heads; rows past the group's heads are zero), B = the K tile through ldmatrix.
// The score accumulators of a head are, element for element, the A fragment of P (heads x rows)
// for the value product O += P V, B = the V tile through ldmatrix.trans.  Scores stay fp32 (fp16 q and
// k, exact products); p enters the value product in fp16 (2^-11 relative per weight).
constexpr int SA_NW = 4;                       // warps per CTA
constexpr int SA_NT = 32 * SA_NW;
constexpr int SA_TR = 16;                      // rows per warp tile
constexpr int SA_TILE = SA_TR * D * 2;         // bytes of one K or V tile (4 KB; a stage holds both)
// tiles per warp in flight or in use: two, so that three CTAs fit an SM (the splits of a launch
// are sized to fill those slots; three stages at two CTAs per SM were 5% slower on lists per kv head)
__host__ __device__ constexpr int sa_stages(int) { return 2; }
__host__ __device__ constexpr int sa_tiles(int nh) { return SA_NW * sa_stages(nh) * 2 * SA_TILE; }  // [warp][stage][K, V]
constexpr int SA_TILES = sa_tiles(1);  // the smaller stage area (the warp states of the merge fit it)
constexpr int SA_REC = 4 + D;
constexpr int SA_NORM_CHUNKS = 8;  // CTAs per (sequence, q head) row of the normalization launch (4: 3% slower)
constexpr int SA_MAX_RPS = 2048;   // rows per split: their offsets are resolved into shared memory

// 16-byte global -> shared copy; a row that is not there reads as zeros
__device__ __forceinline__ void sa_cp16(uint32_t dst, const void* src, bool ok) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(ok ? 16 : 0) : "memory");
}
__device__ __forceinline__ void sa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void sa_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void sa_ldm4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void sa_ldm4t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
// (d0, d1) += A B for an A whose rows 8..15 are zero: a0, a2 are rows 0..7 (k 0..7, 8..15)
__device__ __forceinline__ void sa_mma(float& d0, float& d1, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    [[maybe_unused]] float j2, j3;  // rows 8..15 of the product: not used
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %10, %10};"
        : "+f"(d0), "+f"(d1), "=f"(j2), "=f"(j3)
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.0f));
}
__device__ __forceinline__ uint32_t sa_pack_h2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// byte offset of 16-byte chunk c of tile row r (chunks XOR-swizzled by r mod 8: conflict-free ldmatrix)
__device__ __forceinline__ uint32_t sa_chunk(int r, int c) { return (uint32_t)((r * 16 + (c ^ (r & 7))) * 16); }

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
    float2* fin;        // [batch][H_q] (max, sum) of the exp2 scores, for the probabilities
    KvqWsHeader* hdr;
    int32_t n_splits;
    int32_t rps;        // rows per split (at most)
    int32_t k_target;   // splits per list that fill the resident CTA slots of the launch
    // dense kv heads of a mixed layer: every token is listed (no sel), and only the kv heads g with
    // dense[b][g] != 0 are attended (lists per kv head)
    const int32_t* dense = nullptr;
    int32_t all_tokens = 0;
};

template <int NH>
__global__ void __launch_bounds__(SA_NT) sparse_attn_kernel(SAArgs a) {
    extern __shared__ __align__(16) float sm[];  // warp tiles (then [SA_NW][NH][SA_REC] warp states) | row offsets
    __shared__ int is_last;
    // splits vary slowest over the grid: the first splits of every list, the ones that have rows
    // whatever the lists' lengths, are scheduled first
    const int list = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    // dependent launch: wait for the previous kernel here; let the next one be scheduled only once
    // this CTA's rows are done (an earlier trigger lets a cluster kernel that follows place its
    // CTAs piecemeal while these still hold the SMs)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n_lists = a.per_kv ? a.H : a.H * a.GQ;
    const int Hq = a.H * a.GQ;
    const int g = a.per_kv ? list : list / a.GQ;
    const int h0 = a.per_kv ? list * a.GQ : list;
    int T = a.seq_lens[b];
    if (T > a.max_len) {  // ids are checked against min(seq_len, max_len): the block table's reach
        if (tid == 0 && split == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
        T = a.max_len;
    }
    if (a.dense != nullptr && a.dense[(int64_t)b * a.H + g] == 0) return;  // a sparse kv head: not here
    int n = a.all_tokens ? T : a.sel_count[(int64_t)b * n_lists + list];
    if (n > a.sel_cap || n < 0) {
        if (tid == 0 && split == 0) kvq_dev_flag(a.hdr, KVQ_DEV_OVERFLOW, b);
        n = max(0, min(n, a.sel_cap));
    }
    if (n == 0) {
        if (split == 0)
            for (int i = tid; i < NH * D; i += SA_NT) a.out[((int64_t)b * Hq + h0) * D + i] = 0.0f;
        return;
    }
    // the list's rows in equal shares (whole 16-row tiles) over enough splits to fill the launch's
    // resident CTA slots (k_target per list), at most a.rps rows and at least 64 rows a split: the
    // list is done when its longest share is
    const int k_min = (n + a.rps - 1) / a.rps;
    const int k = min(a.n_splits, max(k_min, min(max(a.k_target, 1), (n + 63) / 64)));
    const int rps_b = ((n + k - 1) / k + SA_TR - 1) / SA_TR * SA_TR;
    const int nsplit_b = (n + rps_b - 1) / rps_b;
    if (split >= nsplit_b) return;
    const int r_begin = split * rps_b, r_end = min(n, r_begin + rps_b);
    const int32_t* ids = a.all_tokens ? nullptr : a.sel + ((int64_t)b * n_lists + list) * a.sel_cap;

    // the split's rows: ids and pages resolved up front into row offsets (in 128-element rows;
    // ~0u for a bad id or page), four per thread in flight
    constexpr int SA_STAGES = sa_stages(NH);
    uint32_t* roff = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(sm) + sa_tiles(NH));
    for (int i0 = r_begin + tid; i0 < r_end; i0 += 4 * SA_NT) {
        int t[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * SA_NT;
            t[u] = i < r_end ? (ids != nullptr ? ids[i] : i) : -1;
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

    const int warp = tid >> 5, lane = tid & 31, hq = lane >> 2, qd = lane & 3;
    // A operand: q rows of the group's heads (fragment row hq), channel pairs 8ks + qd and 8ks + 4 + qd
    uint32_t qa[8][2];
    {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(a.q + ((int64_t)b * Hq + h0 + min(hq, NH - 1)) * D);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            qa[ks][0] = hq < NH ? qrow[8 * ks + qd] : 0u;
            qa[ks][1] = hq < NH ? qrow[8 * ks + 4 + qd] : 0u;
        }
    }
    const int n_tiles = (r_end - r_begin + SA_TR - 1) / SA_TR;
    const uint32_t tiles = (uint32_t)__cvta_generic_to_shared(sm) + (uint32_t)(warp * SA_STAGES * 2 * SA_TILE);
    // tile t of the split (list rows r_begin + 16 t ...) into stage buffer `buf`: K, then V
    auto stage = [&](int t, uint32_t buf) {
        if (t < n_tiles) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int row = (lane >> 4) + 2 * k, c = lane & 15;
                const int i = r_begin + SA_TR * t + row;
                const uint32_t r = i < r_end ? roff[i - r_begin] : 0xffffffffu;
                const bool ok = r != 0xffffffffu;
                const int64_t off = ok ? (int64_t)r * D + 8 * c : 0;
                sa_cp16(buf + sa_chunk(row, c), a.k16 + off, ok);
                sa_cp16(buf + SA_TILE + sa_chunk(row, c), a.v16 + off, ok);
            }
        }
        sa_commit();
    };
    float m = -INFINITY, lsum = 0.0f, o[16][2];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = 0.0f;
    int t = warp;
#pragma unroll
    for (int st = 0; st < SA_STAGES; ++st) stage(t + st * SA_NW, tiles + (uint32_t)(st * 2 * SA_TILE));
    for (int it = 0; t < n_tiles; ++it, t += SA_NW) {  // uniform over the warp
        const uint32_t buf = tiles + (uint32_t)((it % SA_STAGES) * 2 * SA_TILE);
        sa_wait<SA_STAGES - 1>();
        __syncwarp();
        // scores of rows 2qd, 2qd + 1 (n-tile 0) and 8 + 2qd, 9 + 2qd (n-tile 1) for head hq
        float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const int mi = lane >> 3, lr = lane & 7;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t b0, b1, b2, b3;
            sa_ldm4(buf + sa_chunk(lr + 8 * (mi >> 1), 2 * ks + (mi & 1)), b0, b1, b2, b3);
            sa_mma(x[0], x[1], qa[ks][0], qa[ks][1], b0, b1);
            sa_mma(x[2], x[3], qa[ks][0], qa[ks][1], b2, b3);
        }
        const int i0 = r_begin + SA_TR * t;
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + 8 * (j >> 1) + 2 * qd + (j & 1);
            const bool ok = i < r_end && roff[i - r_begin] != 0xffffffffu;
            x[j] = ok ? x[j] * KVQ_SCORE_LOG2_SCALE : -INFINITY;
            mx = fmaxf(mx, x[j]);
            if (a.probs != nullptr && hq < NH && i < r_end) a.probs[((int64_t)b * Hq + h0 + hq) * a.sel_cap + i] = x[j];
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(m, mx);
        float alpha = 1.0f, p[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (mn != -INFINITY) {
            alpha = exp2f(m - mn);
#pragma unroll
            for (int j = 0; j < 4; ++j) p[j] = exp2f(x[j] - mn);
            m = mn;
        }
        lsum = lsum * alpha + ((p[0] + p[1]) + (p[2] + p[3]));
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                o[j][0] *= alpha;
                o[j][1] *= alpha;
            }
        }
        const uint32_t pa0 = sa_pack_h2(p[0], p[1]), pa2 = sa_pack_h2(p[2], p[3]);
#pragma unroll
        for (int nc = 0; nc < 8; ++nc) {
            uint32_t b0, b1, b2, b3;
            sa_ldm4t(buf + SA_TILE + sa_chunk(lr + 8 * (mi & 1), 2 * nc + (mi >> 1)), b0, b1, b2, b3);
            sa_mma(o[2 * nc][0], o[2 * nc][1], pa0, pa2, b0, b1);
            sa_mma(o[2 * nc + 1][0], o[2 * nc + 1][1], pa0, pa2, b2, b3);
        }
        __syncwarp();  // every lane is done with the buffer
        stage(t + SA_STAGES * SA_NW, buf);
    }
    sa_wait<0>();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    // ---- merge the warp states of the CTA (the records reuse the tile buffers)
    __syncthreads();
    if (hq < NH) {
        float* r = sm + (warp * NH + hq) * SA_REC;
        if (qd == 0) {
            r[0] = m;
            r[1] = lsum;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            r[4 + 8 * j + 2 * qd] = o[j][0];
            r[4 + 8 * j + 2 * qd + 1] = o[j][1];
        }
    }
    __syncthreads();
    const int64_t rec0 = (((int64_t)b * n_lists + list) * a.n_splits + split) * NH;
    for (int e = tid; e < NH * D; e += SA_NT) {
        const int hh = e / D, d = e % D;
        float M = -INFINITY;
        for (int w = 0; w < SA_NW; ++w) M = fmaxf(M, sm[(w * NH + hh) * SA_REC]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
            for (int w = 0; w < SA_NW; ++w) {
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
    // ---- last CTA: merge the splits (in parallel over the splits: the heads' max and sum by block
    // reductions, each split's weight kept in shared memory, every warp accumulating all outputs
    // over its share of the splits, the warps' sums added in a fixed order), write the output
    __shared__ float red_m[SA_NW][NH], red_l[SA_NW][NH];
    __shared__ float fin_m[NH], fin_l[NH];
    const float* rec = a.part + ((int64_t)b * n_lists + list) * a.n_splits * NH * SA_REC;  // [split][head]
    float* wsp = sm;                               // [split][head] weights
    float* po = sm + ((nsplit_b * NH + 3) & ~3);   // [warp][head * D + d] partial outputs
    static_assert(NH * D % 32 == 0, "whole warps of outputs");
    float mh[NH];
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) mh[hh] = -INFINITY;
    for (int sp = tid; sp < nsplit_b; sp += SA_NT)
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) mh[hh] = fmaxf(mh[hh], __ldcg(rec + (sp * NH + hh) * SA_REC));
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        float v = mh[hh];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) red_m[warp][hh] = v;
    }
    __syncthreads();
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        float v = red_m[0][hh];
        for (int w = 1; w < SA_NW; ++w) v = fmaxf(v, red_m[w][hh]);
        mh[hh] = v;
    }
    float lh[NH];
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) lh[hh] = 0.0f;
    for (int sp = tid; sp < nsplit_b; sp += SA_NT)
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
            const float* r = rec + (sp * NH + hh) * SA_REC;
            const float w = mh[hh] == -INFINITY ? 0.0f : exp2f(__ldcg(r) - mh[hh]);
            lh[hh] = fmaf(__ldcg(r + 1), w, lh[hh]);
            wsp[sp * NH + hh] = w;
        }
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        float v = lh[hh];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red_l[warp][hh] = v;
    }
    __syncthreads();  // weights and per-warp sums visible
    {
        constexpr int NJ = NH * D / 32;  // outputs per lane: e = lane + 32 j
        float acc[NJ];
#pragma unroll
        for (int j = 0; j < NJ; ++j) acc[j] = 0.0f;
        for (int sp = warp; sp < nsplit_b; sp += SA_NW) {
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int e = lane + 32 * j, hh = e / D, d = e % D;
                acc[j] = fmaf(wsp[sp * NH + hh], __ldcg(rec + (sp * NH + hh) * SA_REC + 4 + d), acc[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < NJ; ++j) po[warp * NH * D + lane + 32 * j] = acc[j];
    }
    if (tid < NH) {  // (the max again from the warps' maxima: no register array indexed by tid)
        float v = 0.0f, m = red_m[0][tid];
        for (int w = 0; w < SA_NW; ++w) {
            v += red_l[w][tid];
            m = fmaxf(m, red_m[w][tid]);
        }
        fin_m[tid] = m;
        fin_l[tid] = v;
    }
    __syncthreads();
    for (int e = tid; e < NH * D; e += SA_NT) {
        const int hh = e / D, d = e % D;
        float O = 0.0f;
        for (int w = 0; w < SA_NW; ++w) O += po[w * NH * D + e];
        const float L = fin_l[hh];
        a.out[((int64_t)b * Hq + h0 + hh) * D + d] = L > 0.0f ? O / L : 0.0f;
    }
    if (tid == 0) a.counters[(int64_t)b * n_lists + list] = 0;
    if (a.probs == nullptr) return;
    if (tid < NH) a.fin[(int64_t)b * Hq + h0 + tid] = make_float2(fin_m[tid], fin_l[tid]);
}

// The stored exp2-domain scores become probabilities, p = 2^(s - max) / sum, one thread per
// (row, q head) with four rows in flight; (max, sum) come from the attention kernel's last CTAs.
__global__ void __launch_bounds__(256) sa_norm_kernel(SAArgs a) {
    kvq_pdl_begin();
    const int h = blockIdx.y, b = blockIdx.z, Hq = a.H * a.GQ;
    const int n_lists = a.per_kv ? a.H : Hq;
    const int list = a.per_kv ? h / a.GQ : h;
    const int n = max(0, min(a.sel_count[(int64_t)b * n_lists + list], a.sel_cap));
    if ((int)blockIdx.x * 1024 >= n) return;
    const float2 f = a.fin[(int64_t)b * Hq + h];
    float* pr = a.probs + ((int64_t)b * Hq + h) * a.sel_cap;
    // 1024-entry chunks, strided over the few CTAs of the row: the grid is sized by the capacity,
    // not by the lists' lengths (on the device), so it stays small
    for (int i0 = blockIdx.x * 1024 + threadIdx.x; i0 < n; i0 += gridDim.x * 1024) {
        float sv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) sv[u] = i0 + 256 * u < n ? __ldcg(pr + i0 + 256 * u) : -INFINITY;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (i0 + 256 * u < n)
                pr[i0 + 256 * u] = (f.y > 0.0f && sv[u] != -INFINITY) ? exp2f(sv[u] - f.x) / f.y : 0.0f;
    }
}

struct SAPlan {
    int n_splits, rps;
};

SAPlan sa_plan(const kvq_layout* L, const kvq_seqs* S, int32_t sel_cap, int per_kv) {
    const int n_lists = per_kv ? L->n_kv_heads : L->n_q_heads;
    const int64_t units = (int64_t)std::max(S->batch, 1) * n_lists;
    const int64_t target = 3LL * kvq_num_sms();  // resident CTAs: one wave, no partial second one
    int splits = (int)std::max<int64_t>(1, target / units);
    int rps = (std::max(sel_cap, 1) + splits - 1) / splits;
    rps = std::min(SA_MAX_RPS, std::max(64, (rps + 63) / 64 * 64));
    splits = (std::max(sel_cap, 1) + rps - 1) / rps;
    return {splits, rps};
}

size_t sa_ws_layout(const kvq_layout* L, const kvq_seqs* S, int32_t sel_cap, size_t* off_part, size_t* off_cnt,
                    size_t* off_fin) {
    // sized for the larger of the two list modes so one workspace serves both
    const SAPlan p0 = sa_plan(L, S, sel_cap, 0), p1 = sa_plan(L, S, sel_cap, 1);
    const int GQ = L->n_q_heads / std::max(L->n_kv_heads, 1);
    const size_t r0 = (size_t)std::max(S->batch, 1) * L->n_q_heads * p0.n_splits;
    const size_t r1 = (size_t)std::max(S->batch, 1) * L->n_kv_heads * p1.n_splits * GQ;
    const size_t recs = r0 > r1 ? r0 : r1;
    *off_part = sizeof(KvqWsHeader);
    *off_cnt = kvq_round_up(*off_part + recs * SA_REC * sizeof(float), 256);
    *off_fin = kvq_round_up(*off_cnt + (size_t)std::max(S->batch, 1) * L->n_q_heads * sizeof(int32_t), 256);
    return kvq_round_up(*off_fin + (size_t)std::max(S->batch, 1) * L->n_q_heads * sizeof(float2), 256);
}

template <int NH>
int launch_sa(const SAArgs& a, dim3 grid, cudaStream_t s, bool pdl = true) {
    static_assert((size_t)SA_NW * 8 * SA_REC * sizeof(float) <= (size_t)SA_TILES, "the warp states fit the tiles");
    const size_t smem = (size_t)sa_tiles(NH) + (size_t)a.rps * sizeof(uint32_t);
    const int st = kvq_prepare_kernel((const void*)sparse_attn_kernel<NH>,
                                      (int)((size_t)sa_tiles(NH) + SA_MAX_RPS * sizeof(uint32_t)));
    if (st) return st;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sparse_attn_kernel<NH>, SA_NT, smem) != cudaSuccess)
        occ = 1;
    SAArgs b = a;
    const int64_t units = (int64_t)grid.x * grid.z;
    b.k_target = (int)std::max<int64_t>(1, (int64_t)std::max(occ, 1) * kvq_num_sms() / std::max<int64_t>(units, 1));
    // a dependent launch (it may be scheduled while the previous kernel finishes), except after the
    // mixed layer's cluster kernel, whose early trigger would only queue these CTAs behind it
    if (!pdl) {
        sparse_attn_kernel<NH><<<grid, SA_NT, smem, s>>>(b);
        return kvq_launch_status("kv_sparse_attn");
    }
    const cudaError_t e = kvq_launch_pdl(sparse_attn_kernel<NH>, grid, dim3(SA_NT), smem, s, b);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_sparse_attn launch: %s", cudaGetErrorString(e));
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

template <int NHS>
int launch_crit_nhs(CritArgs& a, const kvq_layout* L, const kvq_seqs* S, cudaStream_t s) {
    const int st = kvq_prepare_kernel((const void*)crit_score_kernel<NHS>, 0);
    if (st) return st;
    a.tiles = std::max(1, (S->max_len + CS_TILE - 1) / CS_TILE);
    a.n_items = S->batch * (NHS == 1 ? L->n_q_heads : L->n_kv_heads) * a.tiles;
    const int grid = std::min(a.n_items, kvq_num_sms() * (NHS <= 2 ? CS_MINB : 2));
    crit_score_kernel<NHS><<<grid, CS_NT, 0, s>>>(a);
    return KVQ_OK;
}

// group == false: one score row per q head; true: one row per kv head, its q heads summed.
int launch_crit(CritArgs& a, const kvq_layout* L, const kvq_seqs* S, cudaStream_t s, bool group = false) {
    switch (group ? a.GQ : 1) {
        case 2: return launch_crit_nhs<2>(a, L, S, s);
        case 4: return launch_crit_nhs<4>(a, L, S, s);
        case 8: return launch_crit_nhs<8>(a, L, S, s);
        default: return launch_crit_nhs<1>(a, L, S, s);
    }
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

extern "C" int kv_group_critical_score(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q,
                                       int32_t n_crit, int32_t* crit, float* scores, int64_t score_stride,
                                       void* stream) {
    kvq_clear_error();
    int st = crit_common(L, P, S, q, n_crit, scores, score_stride, "kv_group_critical_score");
    if (st) return st;
    if (S->batch == 0) return KVQ_OK;
    CritArgs a = crit_args(L, P, S, q, n_crit, crit, scores, score_stride);
    st = launch_crit(a, L, S, kvq_stream(stream), true);
    if (st) return st;
    return kvq_launch_status("kv_group_critical_score");
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

// The dense kv heads of a mixed layer (kv_mixed_layer_decode's second launch): exact attention of each
// dense kv head's q heads over every cached token, lists per kv head with the group's heads sharing
// each staged K/V tile; sparse kv heads' CTAs return at once.  The workspace is kv_sparse_attn's
// for sel_cap = max_len.
// Splits of the all-tokens mode: at most 1024 rows each (a warp then walks at most 16 staged
// tiles), at least 64 rows
static SAPlan sa_plan_all(const kvq_seqs* S) {
    const int cap = std::max(S->max_len, 1);
    const int rps = std::min(1024, std::max(64, ((cap + 127) / 128 + 63) / 64 * 64));
    return {(cap + rps - 1) / rps, rps};
}

static size_t dense_ws_layout(const kvq_layout* L, const kvq_seqs* S, size_t* off_part, size_t* off_cnt, size_t* off_fin) {
    const SAPlan p = sa_plan_all(S);
    const int GQ = L->n_q_heads / std::max(L->n_kv_heads, 1);
    const size_t recs = (size_t)std::max(S->batch, 1) * L->n_kv_heads * p.n_splits * GQ;
    *off_part = sizeof(KvqWsHeader);
    *off_cnt = kvq_round_up(*off_part + recs * SA_REC * sizeof(float), 256);
    *off_fin = kvq_round_up(*off_cnt + (size_t)std::max(S->batch, 1) * L->n_q_heads * sizeof(int32_t), 256);
    return kvq_round_up(*off_fin + (size_t)std::max(S->batch, 1) * L->n_q_heads * sizeof(float2), 256);
}

size_t kvq_dense_heads_attn_ws(const kvq_layout* L, const kvq_seqs* S) {
    size_t a, c, f;
    return dense_ws_layout(L, S, &a, &c, &f);
}

int kvq_dense_heads_attn(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q,
                         const int32_t* dense, float* out, void* ws, cudaStream_t s) {
    size_t off_part, off_cnt, off_fin;
    const int32_t cap = std::max(S->max_len, 1);
    dense_ws_layout(L, S, &off_part, &off_cnt, &off_fin);
    const SAPlan p = sa_plan_all(S);
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
    a.sel = nullptr;
    a.sel_cap = cap;
    a.sel_count = nullptr;
    a.per_kv = 1;
    a.out = out;
    a.probs = nullptr;
    a.part = reinterpret_cast<float*>(static_cast<char*>(ws) + off_part);
    a.counters = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + off_cnt);
    a.fin = reinterpret_cast<float2*>(static_cast<char*>(ws) + off_fin);
    a.hdr = static_cast<KvqWsHeader*>(ws);
    a.n_splits = p.n_splits;
    a.rps = p.rps;
    a.dense = dense;
    a.all_tokens = 1;
    const dim3 grid(L->n_kv_heads, p.n_splits, S->batch);
    switch (a.GQ) {
        case 1: return launch_sa<1>(a, grid, s, false);
        case 2: return launch_sa<2>(a, grid, s, false);
        case 4: return launch_sa<4>(a, grid, s, false);
        default: return launch_sa<8>(a, grid, s, false);
    }
}

extern "C" size_t kv_sparse_attn_ws(const kvq_layout* L, const kvq_seqs* S, int32_t sel_cap) {
    if (kvq_check_layout(L, "kv_sparse_attn_ws", true) || kvq_check_seqs_sizes(S, "kv_sparse_attn_ws") || sel_cap <= 0)
        return 0;
    size_t a, c, f;
    return sa_ws_layout(L, S, sel_cap, &a, &c, &f);
}

// kv_sparse_attn without its normalization launch: probs (when given) keeps the log2-domain scores
// and the workspace the (max, sum) per (sequence, q head) that make them probabilities.
static int sparse_attn_scores(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q,
                              const int32_t* sel, int32_t sel_cap, const int32_t* sel_count, int32_t sel_per_kv_head,
                              float* out, float* probs, void* ws, size_t ws_bytes, void* stream) {
    int st = kvq_check_layout(L, "kv_sparse_attn", true);
    if (st) return st;
    st = kvq_check_seqs(S, "kv_sparse_attn");
    if (st) return st;
    KVQ_REQUIRE(P && P->k16 && P->v16, KVQ_ERR_INVALID_ARG, "kv_sparse_attn: pool needs k16 and v16");
    KVQ_REQUIRE(((uintptr_t)P->k16 & 15u) == 0 && ((uintptr_t)P->v16 & 15u) == 0, KVQ_ERR_INVALID_ARG,
                "kv_sparse_attn: k16/v16 must be 16-byte aligned");
    KVQ_REQUIRE(sel_cap > 0 && sel && sel_count && out, KVQ_ERR_INVALID_ARG, "kv_sparse_attn: NULL buffer or sel_cap");
    KVQ_REQUIRE(sel_per_kv_head == 0 || sel_per_kv_head == 1, KVQ_ERR_INVALID_ARG, "kv_sparse_attn: sel_per_kv_head");
    size_t off_part, off_cnt, off_fin;
    const size_t need = sa_ws_layout(L, S, sel_cap, &off_part, &off_cnt, &off_fin);
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
    a.fin = reinterpret_cast<float2*>(static_cast<char*>(ws) + off_fin);
    a.hdr = static_cast<KvqWsHeader*>(ws);
    a.n_splits = p.n_splits;
    a.rps = p.rps;
    const int n_lists = sel_per_kv_head ? L->n_kv_heads : L->n_q_heads;
    dim3 grid(n_lists, p.n_splits, S->batch);
    cudaStream_t s = kvq_stream(stream);
    int e;
    if (!sel_per_kv_head) {
        e = launch_sa<1>(a, grid, s);
    } else {
        switch (a.GQ) {
            case 1: e = launch_sa<1>(a, grid, s); break;
            case 2: e = launch_sa<2>(a, grid, s); break;
            case 4: e = launch_sa<4>(a, grid, s); break;
            default: e = launch_sa<8>(a, grid, s); break;
        }
    }
    return e;
}

extern "C" int kv_sparse_attn(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q,
                              const int32_t* sel, int32_t sel_cap, const int32_t* sel_count, int32_t sel_per_kv_head,
                              float* out, float* probs, void* ws, size_t ws_bytes, void* stream) {
    kvq_clear_error();
    const int e = sparse_attn_scores(L, P, S, q, sel, sel_cap, sel_count, sel_per_kv_head, out, probs, ws, ws_bytes,
                                     stream);
    if (e || probs == nullptr || S->batch == 0) return e;
    // the stored scores become probabilities (a second, short launch)
    size_t off_part, off_cnt, off_fin;
    sa_ws_layout(L, S, sel_cap, &off_part, &off_cnt, &off_fin);
    SAArgs a{};
    a.H = L->n_kv_heads;
    a.GQ = L->n_q_heads / L->n_kv_heads;
    a.sel_cap = sel_cap;
    a.sel_count = sel_count;
    a.per_kv = sel_per_kv_head;
    a.probs = probs;
    a.fin = reinterpret_cast<float2*>(static_cast<char*>(ws) + off_fin);
    const dim3 ng((unsigned)std::min((sel_cap + 1023) / 1024, SA_NORM_CHUNKS), (unsigned)L->n_q_heads, (unsigned)S->batch);
    const int st2 = kvq_prepare_kernel((const void*)sa_norm_kernel, 0);
    if (st2) return st2;
    const cudaError_t le = kvq_launch_pdl(sa_norm_kernel, ng, dim3(256), 0, kvq_stream(stream), a);
    if (le != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_sparse_attn launch: %s", cudaGetErrorString(le));
    return kvq_launch_status("kv_sparse_attn");
}
