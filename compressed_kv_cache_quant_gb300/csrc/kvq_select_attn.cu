// a5 kv_topk_select and the fused a5+a6 kv_select_sparse_attn.
//
// [TailorKV §2.3, §5.1] keep the k tokens with the highest approximate score,
// [KVSurvey §三.1] always keep the attention sinks and the recent window;
// [Meeting §3.2] exact softmax attention over the kept tokens.
//
// One cluster of 8 CTAs serves one (sequence, query head).  CTA r owns the
// r-th eighth of the positions and holds their order-preserving 32-bit keys
// in shared memory.  The k-th largest key is found by radix selection with a
// 12-bit first digit (taken from the per-head histogram the score kernel
// accumulated, or built here) and two 10-bit digits over the few candidates
// that share the first digit; partial histograms are summed through
// distributed shared memory.  Ties at the k-th key go to the lower positions
// (a cluster-wide prefix count).  The kept positions are compacted in order;
// each CTA then attends its own kept rows and the 8 partial softmax states are
// merged by log-sum-exp in rank 0.
#include <cooperative_groups.h>

#include <algorithm>
#include <cstddef>

#include "kvq_internal.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int D = KVQ_HEAD_DIM;
constexpr int PG = KVQ_BLOCK_TOKENS;
constexpr int CL = 8;                 // CTAs per cluster
constexpr int NT = 512;               // threads per CTA
constexpr int NW = NT / 32;
constexpr int MAX_CHUNK = 45056;      // positions per CTA (keys in shared memory)
constexpr int MAXIT = (MAX_CHUNK + NT - 1) / NT;  // 32-position steps per warp in the compaction
constexpr int H1 = 4096;              // first digit: key bits 31..20
constexpr int H2 = 1024;              // second and third digits: bits 19..10, 9..0
constexpr int NHW = NT / 16;          // half-warps (attention: one row per half-warp)
constexpr int BATCH = 4;              // rows in flight per half-warp
constexpr int PF_ALL_MAX = 1024;      // kept rows per CTA prefetched to L2 before the attention
constexpr int PF_AHEAD = 2;           // longer lists: rows prefetched this many batches ahead
constexpr int REC = 4 + D;
constexpr uint32_t ROW_NONE = 0xffffffffu;  // attention row ids: no row
constexpr uint32_t ROW_NEW = 0xfffffffeu;   // the newest token, read from k_new / v_new

struct SXArgs {
    const float* scores;
    int64_t score_stride;
    uint32_t* hist;          // [B][n_heads][4096] or NULL
    const int32_t* seq_lens;
    int32_t max_len;
    int32_t n_heads;
    int32_t k_fixed;
    double ratio;
    int32_t n_sink, window;
    int32_t* sel;            // [B][n_heads][sel_cap] or NULL
    int32_t sel_cap;
    int32_t* sel_count;      // [B][n_heads] or NULL
    KvqWsHeader* hdr;
    // attention (q == NULL: selection only)
    const uint16_t* q;
    const uint16_t* k16;
    const uint16_t* v16;
    int64_t num_blocks;
    const int32_t* bt;
    int32_t max_blocks;
    int32_t H, GQ;
    float* out;
    // fused critical scores (kT != NULL): the keys are computed here from the
    // channel-major K copy after appending the newest token, instead of read
    uint16_t* kT;
    float* absmax;
    int32_t t_cap;
    int32_t n_crit;
    const uint16_t* k_new;
    const uint16_t* v_new;
    uint16_t* k16w;
    uint16_t* v16w;
    float* scores_out;       // optional copy of the scores [B][H_q][score_stride]
    const int32_t* dense;    // [B][H_kv] (or NULL): non-zero = the kv head's q heads attend every token
    int32_t dense_elsewhere; // dense heads: append and list only (their attention is a second launch)
};

constexpr int CAP_S = 1024;           // kept positions collected per CTA in the one-pass path
constexpr int CAP_C = 512;            // first-digit candidates collected per CTA
static_assert(CL * CAP_C == H1 && CAP_C == NT, "candidate slots: one per thread and rank");

// Shared state of one CTA; it follows the chunk's keys in dynamic shared memory.
struct SXSmem {
    union {
        uint32_t hist[H1];                  // this CTA's first-digit histogram
        uint32_t cand[CL * CAP_C];          // every rank's first-digit candidates (key bits 19..0), CAP_C slots each
    } u;
    union {
        uint32_t gh[H1];                    // the cluster's first-digit histogram
        struct {
            uint32_t h2[H2];                // second digit histogram
            uint32_t h2b[H2];               // third digit histogram (fast path)
            unsigned long long cl[CAP_C];   // this CTA's first-digit candidates
            uint32_t wmask[NW][MAXIT];      // ballots of the ordered compaction
        } w;
        float scratch[NHW * REC];           // half-warp softmax states (attention)
    } v;
    uint32_t list[CAP_S];                   // kept positions, then their row offsets
    uint32_t wsum[NW];
    uint32_t wtot[NW], wtot2[NW];
    uint32_t ncand[CL];                     // first-digit candidates of each rank (above CAP_C: overflow)
    int32_t n_s, n_c;                       // this CTA's kept positions / candidates
    uint32_t nsc;                           // both, packed (low / high 16 bits) while classifying
    int32_t bc_cut;
    uint32_t s_bin, s_above;
    uint32_t eq_cnt, sel_cnt;               // this CTA's counts, read by the others
    float st_m[CL], st_l[CL];               // rank 0: the CTAs' softmax states
    float st_o[CL][D];
    uint32_t eqr[CL];                       // candidates equal to the k-th key, per owner rank
    uint32_t sml[32], nsm;                  // candidates sharing the second digit (short list)
    float qs[D];                            // fused scores: the query
    unsigned long long ck[D];               // channel importance key | (255 - channel)
    uint32_t crank[D];                      // its rank among the channels
    uint16_t knew[D];
    int32_t clist[D];
};

size_t smem_bytes(int chunk) { return kvq_round_up((size_t)std::max(chunk, 1) * sizeof(uint32_t), 16) + sizeof(SXSmem); }
int chunk_of(int T) { return ((T + CL - 1) / CL + 31) / 32 * 32; }
__device__ __forceinline__ int chunk_of_dev(int T) { return ((T + CL - 1) / CL + 31) / 32 * 32; }

// A cluster barrier split in two: arrive (releasing this thread's earlier writes) early, wait
// (acquiring the other CTAs' writes) where they are needed.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

template <int N>
__device__ __forceinline__ uint32_t excl_scan(uint32_t v, uint32_t* wsum, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < N / 32 ? wsum[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < N / 32) wsum[lane] = w;
    }
    __syncthreads();
    *total = wsum[N / 32 - 1];
    return x - v + (warp > 0 ? wsum[warp - 1] : 0u);
}

// Over the NT * PER bins in tot[], finds the bin (from the top) that holds the `remaining`-th
// largest element: s.s_bin, and s.s_above = the count in higher bins.  Called by a whole CTA;
// warp w owns 32 * PER consecutive bins (warp 0 the highest), lane l PER of them; two barriers.
template <int PER>
__device__ __forceinline__ void find_bin_from_top(const uint32_t* tot, uint32_t remaining, SXSmem& s) {
    constexpr int NB = NT * PER;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int top = NB - 32 * PER * warp - PER * lane;  // this lane's bins: top - PER .. top - 1
    uint32_t c[PER], mine = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        c[j] = tot[top - 1 - j];
        mine += c[j];
    }
    uint32_t x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s.wsum[warp] = x;
    __syncthreads();
    uint32_t before = 0;
    int ws = -1;
    for (int w = 0; w < NW; ++w) {
        const uint32_t t = s.wsum[w];
        if (before + t >= remaining) {
            ws = w;
            break;
        }
        before += t;
    }
    if (warp == ws) {
        uint32_t run = before + x - mine;  // the count above this lane's bins
        if (run < remaining && run + mine >= remaining) {
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                if (run + c[j] >= remaining) {
                    s.s_bin = (uint32_t)(top - 1 - j);
                    s.s_above = run;
                    break;
                }
                run += c[j];
            }
        }
    }
    __syncthreads();
}

__device__ __forceinline__ void unpack8(const uint4& r, float* f) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}

// Starts pulling the 256-byte row at p (256-byte aligned) into L2; no completion to wait for.
__device__ __forceinline__ void prefetch_row_l2(const void* p) {
    const char* c = static_cast<const char*>(p);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(c) : "memory");
    asm volatile("prefetch.global.L2 [%0];" ::"l"(c + 128) : "memory");
}

// Row offset (in 128-element rows) of position t of kv head g of sequence b on page `page`; ROW_NEW
// for the newest token (read from its source), ROW_NONE (flagged) for a page outside the pool.
__device__ __forceinline__ uint32_t row_of(const SXArgs& a, int b, int g, int t, int t_new, int32_t page) {
    if (t == t_new) return ROW_NEW;
    if (page >= 0 && page < a.num_blocks) return (uint32_t)(((int64_t)page * a.H + g) * PG + (t & 15));
    kvq_dev_flag(a.hdr, KVQ_DEV_BAD_PAGE, t);
    return ROW_NONE;
}

// acc[i] += q_c * K[p0 + i][c] for the 8 positions in `raw` (fp16); position p0 + inew is
// the newest token, whose key `knew` is not in the channel-major copy's load yet.
__device__ __forceinline__ void score_channel(const uint4& raw, float qc, bool has_new, int inew, uint16_t knew,
                                              float* acc) {
    float kf[8];
    unpack8(raw, kf);
    if (has_new) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (inew == i) kf[i] = kvq_h2f(knew);
    }
    // fma == add of the exact fp16*fp16 product: the same fp32 result as (q*k) + acc
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = fmaf(qc, kf[i], acc[i]);
}

// The 8 scores of positions p0.. (those below hi): their keys into the chunk's key array, the
// candidates' first digits into the local histogram, the scores to srow_out if given.
__device__ __forceinline__ void score_finish(const float* acc, int p0, int lo, int hi, int cand_lo, int cand_hi,
                                             uint32_t* keys, uint32_t* hist, float* srow_out) {
    if (srow_out != nullptr) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (p0 + i < hi) srow_out[p0 + i] = acc[i];
    }
    const bool full = p0 + 8 <= hi;
#pragma unroll
    for (int h4 = 0; h4 < 8; h4 += 4) {  // four keys at a time: fewer live registers
        uint32_t kk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            kk[i] = kvq_float_key(acc[h4 + i]);
            const int p = p0 + h4 + i;
            if (p < hi && p >= cand_lo && p < cand_hi) atomicAdd(&hist[kk[i] >> 20], 1u);
        }
        if (full) {
            *reinterpret_cast<uint4*>(keys + (p0 - lo) + h4) = make_uint4(kk[0], kk[1], kk[2], kk[3]);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (p0 + h4 + i < hi) keys[p0 + h4 + i - lo] = kk[i];
        }
    }
}

// Second phase of the classification, one queued group of eight keys per lane (has = false:
// none): entry = chunk offset << 8 | mask of the keys at or above bin b1 or outside the
// candidate range.  Those above the bin or outside the range are kept (s.list), those in the
// bin are candidates (s.v.w.cl, with their keys); both counts are reserved with one packed
// atomic per warp (each stays below the chunk size < 65536: no carry between the halves).
__device__ __forceinline__ void classify_group(bool has, uint32_t e, const uint32_t* keys, int lo, int cand_lo,
                                               int cand_hi, uint32_t hi_thr, SXSmem& s, int lane) {
    const int q0 = has ? (int)(e >> 8) : 0;
    const uint32_t m = has ? (e & 0xffu) : 0u;
    const uint4 ka = *reinterpret_cast<const uint4*>(keys + q0);
    const uint4 kb = *reinterpret_cast<const uint4*>(keys + q0 + 4);
    const uint32_t kk[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
    uint32_t fs = 0u, fc = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (!((m >> i) & 1u)) continue;
        const int p = lo + q0 + i;
        if (p < cand_lo || p >= cand_hi || kk[i] > hi_thr) fs |= 1u << i;
        else fc |= 1u << i;
    }
    const uint32_t cnt = (uint32_t)__popc(fs) | ((uint32_t)__popc(fc) << 16);
    uint32_t x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    const uint32_t tot = __shfl_sync(0xffffffffu, x, 31);
    uint32_t bases = 0u;
    if (lane == 0 && tot != 0u) bases = atomicAdd(&s.nsc, tot);
    bases = __shfl_sync(0xffffffffu, bases, 0) + x - cnt;
    uint32_t bs = bases & 0xffffu, bc = bases >> 16;
    const uint32_t p0 = (uint32_t)(lo + q0);
    while (fs) {
        const int i = __ffs(fs) - 1;
        fs &= fs - 1u;
        if (bs < (uint32_t)CAP_S) s.list[bs] = p0 + i;
        ++bs;
    }
    while (fc) {
        const int i = __ffs(fc) - 1;
        fc &= fc - 1u;
        uint32_t key = kk[0];
#pragma unroll
        for (int j = 1; j < 8; ++j) key = i == j ? kk[j] : key;
        if (bc < (uint32_t)CAP_C) s.v.w.cl[bc] = ((unsigned long long)key << 32) | (p0 + i);
        ++bc;
    }
}

// Appends, in ballot order, the lanes with f set to list[*n] (capacity cap);
// returns false if the list overflowed.
template <typename V>
__device__ __forceinline__ bool warp_append(bool f, V v, V* list, int32_t* n, int cap, int lane) {
    const uint32_t m = __ballot_sync(0xffffffffu, f);
    if (m == 0u) return true;
    int base = 0;
    if (lane == 0) base = atomicAdd(n, __popc(m));
    base = __shfl_sync(0xffffffffu, base, 0);
    const int i = base + __popc(m & ((1u << lane) - 1u));
    if (f && i < cap) list[i] = v;
    return base + __popc(m) <= cap;
}

// MODE 1 (lean): the instance for the fused decode without optional outputs (kT given, no sel,
// scores_out or hist, at most 8 critical channels; dense flags allowed).  MODE 2: selection only
// (scores read from memory, no attention, no dense flags).  MODE 0: every option.  The paths an
// instance never takes are not compiled in, so that the instructions a CTA runs once, phase after
// phase, are fetched from fewer lines.
template <int MODE>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(NT, 2) select_attn_kernel(SXArgs a, int chunk_cap) {
    constexpr bool LEAN = MODE == 1, SEL_ONLY = MODE == 2;
    extern __shared__ __align__(16) uint32_t keys[];  // the chunk's keys; later its kept positions
    SXSmem& s = *reinterpret_cast<SXSmem*>(reinterpret_cast<char*>(keys) +
                                           kvq_round_up((size_t)max(chunk_cap, 1) * sizeof(uint32_t), 16));
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = (int64_t)b * a.n_heads + h;
    if constexpr (SEL_ONLY) {
        // wait for the previous kernel; the next one (an attention over the selection) is scheduled
        // when this grid exits: an early trigger would let its CTAs hold SMs beside these clusters
        asm volatile("griddepcontrol.wait;" ::: "memory");
    } else {
        kvq_pdl_begin();
    }
    const bool fused = LEAN || (!SEL_ONLY && a.kT != nullptr);
    // the fused path's per-channel inputs are requested together with the length
    uint16_t pre_q = 0, pre_kn = 0;
    float pre_am = 0.0f;
    if (fused && tid < D) {
        const int64_t kvrow = (int64_t)b * a.H + h / a.GQ;
        pre_q = a.q[row * D + tid];
        pre_am = a.absmax[kvrow * D + tid];
        pre_kn = a.k_new[kvrow * D + tid];
    }
    int T = a.seq_lens[b];
    if (T < 0 || T > a.max_len) {
        if (tid == 0 && rank == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
        T = T < 0 ? 0 : a.max_len;
    }
    const int k = a.k_fixed >= 0 ? a.k_fixed : (int)floor(a.ratio * (double)T);
    const int chunk = chunk_of_dev(T);  // a multiple of 32: the chunk starts 16-byte aligned
    const int lo = min(T, rank * chunk), hi = min(T, lo + chunk);
    const int n = hi - lo;
    // a dense head (head-level classification: quantization-friendly) attends every token: no
    // critical scores, no selection -- the same launch, dispatched by the head's class
    const bool dense = !SEL_ONLY && a.dense != nullptr && a.dense[(int64_t)b * a.H + h / a.GQ] != 0;
    const bool keep_all = dense || (int64_t)T <= (int64_t)a.n_sink + a.window + k;
    const int cand_lo = a.n_sink, cand_hi = T - a.window;
    const float* srow = a.scores + row * a.score_stride;
    // warp w owns the contiguous run [w_lo, w_hi) of the chunk in the ordered passes
    const int wlen = ((n + NW - 1) / NW + 31) / 32 * 32;
    const int w_lo = min(hi, lo + warp * wlen), w_hi = min(hi, w_lo + wlen);
    if (tid == 0) {
        s.n_s = 0;
        s.n_c = 0;
    }
    // the first-digit histograms of the cluster's CTAs are summed into every CTA's copy; the copy is
    // zeroed and the cluster barrier's arrive released where this CTA has no load in flight (a
    // release waits for them), the matching wait precedes the first remote add
    const bool exchange = !keep_all && k > 0 && (fused || a.hist == nullptr);
    const bool has_sel = !LEAN && a.sel != nullptr;
    const bool has_hist = !LEAN && a.hist != nullptr;

    uint32_t kth = 0xffffffffu;  // kept: key > kth, or key == kth and position <= cut
    int32_t cut = -1;
    bool listed = false;         // s.list holds this CTA's kept positions (the one-pass path)
    int n_early = 0;             // s.list[0, n_early) already hold row offsets (rows in flight to L2)
    const int gkv = a.q != nullptr ? h / a.GQ : 0;            // kv head of the attention
    const int t_new = a.k_new != nullptr ? T - 1 : -1;        // the newest token: read from its source
    if (fused) {
        // ---- critical channels [TailorKV §2.3]: s_c = |q_c| max_t |K_c| with the newest token
        // included; the n_crit largest (ties -> lower channel), kept in ascending order
        const int g = h / a.GQ;
        const int64_t kvrow = (int64_t)b * a.H + g;
        const int p_new = T - 1;
        if (tid < D) {
            const float qv = kvq_h2f(pre_q);
            float am = pre_am;
            if (p_new >= 0) {
                const uint16_t kn = pre_kn;
                s.knew[tid] = kn;
                am = fmaxf(am, fabsf(kvq_h2f(kn)));
                if (rank == 0 && h % a.GQ == 0) {
                    // append the newest token of kv head g (one CTA per kv head does it)
                    const int32_t page = a.bt[(int64_t)b * a.max_blocks + (p_new >> 4)];
                    if (page >= 0 && page < a.num_blocks) {
                        const int64_t off = ((page * (int64_t)a.H + g) * PG + (p_new & 15)) * D + tid;
                        a.k16w[off] = kn;
                        a.v16w[off] = a.v_new[kvrow * D + tid];
                    } else {
                        kvq_dev_flag(a.hdr, KVQ_DEV_BAD_PAGE, b);
                    }
                    if (p_new < a.t_cap) a.kT[(kvrow * D + tid) * a.t_cap + p_new] = kn;
                    a.absmax[kvrow * D + tid] = am;
                }
            }
            s.qs[tid] = qv;
            // |q_c| max|K_c|: a product of two fp16 values, exact in fp32; ties -> lower channel
            s.ck[tid] = ((unsigned long long)kvq_float_key(fabsf(qv) * am) << 8) | (unsigned)(255 - tid);
            s.crank[tid] = 0u;
        }
        if (dense && a.dense_elsewhere) {
            // a dense kv head of a mixed layer: appended above; its attention is the second launch.
            // The ordered selection lists every token: position p at entry p (this CTA's chunk)
            if (has_sel) {
                int32_t* outl = a.sel + row * a.sel_cap;
                for (int p = lo + tid; p < hi; p += NT) {
                    if (p < a.sel_cap) outl[p] = p;
                    else kvq_dev_flag(a.hdr, KVQ_DEV_OVERFLOW, b);
                }
                if (rank == 0 && tid == 0 && a.sel_count != nullptr) a.sel_count[row] = min(T, a.sel_cap);
            }
            return;  // uniform over the cluster: no cluster barrier is pending
        }
        for (int i = tid; i < H1; i += NT) s.u.hist[i] = 0u;
        __syncthreads();
        {
            // rank of channel c = number of channels with a larger key; four threads per channel
            static_assert(NT == 4 * D, "four threads per channel");
            const int c = tid & (D - 1), part = tid >> 7;
            const unsigned long long v = s.ck[c];
            uint32_t r = 0;
#pragma unroll 8
            for (int j = 0; j < D / 4; ++j) r += s.ck[part * (D / 4) + j] > v;
            atomicAdd(&s.crank[c], r);
        }
        __syncthreads();
        if (warp == 0) {  // the n_crit channels of rank < n_crit, ascending
            int before = 0;
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
                const int c = lane + 32 * j;
                const bool sel = s.crank[c] < (uint32_t)a.n_crit;
                const uint32_t m = __ballot_sync(0xffffffffu, sel);
                if (sel) s.clist[before + __popc(m & ((1u << lane) - 1u))] = c;
                before += __popc(m);
            }
        }
        __syncthreads();
        // ---- approximate scores a_t = sum over the channels, ascending, of q_c K[t][c] (fp32 from
        // +0), their keys, and the local histogram of candidate keys (a dense head has none)
        if (exchange) {
            for (int i = tid; i < H1; i += NT) s.v.gh[i] = 0u;
            cluster_arrive();
        }
        const uint16_t* kbase = a.kT + kvrow * D * a.t_cap;
        float* srow_out = (!LEAN && a.scores_out != nullptr) ? a.scores_out + row * a.score_stride : nullptr;
        if (dense) {
        } else if (LEAN || a.n_crit <= 8) {
            // one 16-byte load per channel and 8 positions; a channel's registers are refilled
            // with the next group's load as soon as they are consumed, so loads stay in flight
            // channel row offsets: c * t_cap < 128 * 360448 fits in 32 bits
            const uint32_t tcap = (uint32_t)a.t_cap;
            uint4 raw[8];
            int p0 = lo + 8 * tid;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                raw[j] = make_uint4(0u, 0u, 0u, 0u);
                if (j < a.n_crit && p0 < hi)
                    raw[j] = __ldg(reinterpret_cast<const uint4*>(kbase + (uint32_t)s.clist[j] * tcap + p0));
            }
            for (; p0 < hi; p0 += 8 * NT) {
                const int pn = p0 + 8 * NT;
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
                const bool has_new = p_new >= p0 && p_new < p0 + 8;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j >= a.n_crit) break;
                    const int c = s.clist[j];
                    score_channel(raw[j], s.qs[c], has_new, p_new - p0, s.knew[c], acc);
                    if (pn < hi) raw[j] = __ldg(reinterpret_cast<const uint4*>(kbase + (uint32_t)c * tcap + pn));
                }
                score_finish(acc, p0, lo, hi, cand_lo, cand_hi, keys, s.u.hist, srow_out);
            }
        } else {
            for (int p0 = lo + 8 * tid; p0 < hi; p0 += 8 * NT) {
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
                const bool has_new = p_new >= p0 && p_new < p0 + 8;
                for (int j0 = 0; j0 < a.n_crit; j0 += 8) {
                    uint4 raw[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (j0 + j < a.n_crit)
                            raw[j] = __ldg(reinterpret_cast<const uint4*>(kbase + (int64_t)s.clist[j0 + j] * a.t_cap + p0));
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (j0 + j >= a.n_crit) break;
                        const int c = s.clist[j0 + j];
                        score_channel(raw[j], s.qs[c], has_new, p_new - p0, s.knew[c], acc);
                    }
                }
                score_finish(acc, p0, lo, hi, cand_lo, cand_hi, keys, s.u.hist, srow_out);
            }
        }
        __syncthreads();
    }
    if (!keep_all) {
        if (!fused) {
            if (exchange) {
                for (int i = tid; i < H1; i += NT) s.v.gh[i] = 0u;
                cluster_arrive();
            }
            // ---- the chunk's keys (16-byte loads, eight in flight per thread)
            for (int p0 = lo + 4 * tid; p0 < hi; p0 += 4 * NT * 8) {
                float4 v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int p = p0 + j * 4 * NT;
                    if (p + 3 < hi) {
                        v[j] = __ldcg(reinterpret_cast<const float4*>(srow + p));
                    } else {
                        v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (p < hi) v[j].x = srow[p];
                        if (p + 1 < hi) v[j].y = srow[p + 1];
                        if (p + 2 < hi) v[j].z = srow[p + 2];
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int p = p0 + j * 4 * NT;
                    if (p + 3 < hi) {
                        *reinterpret_cast<uint4*>(keys + (p - lo)) =
                            make_uint4(kvq_float_key(v[j].x), kvq_float_key(v[j].y), kvq_float_key(v[j].z),
                                       kvq_float_key(v[j].w));
                    } else {
                        if (p < hi) keys[p - lo] = kvq_float_key(v[j].x);
                        if (p + 1 < hi) keys[p + 1 - lo] = kvq_float_key(v[j].y);
                        if (p + 2 < hi) keys[p + 2 - lo] = kvq_float_key(v[j].z);
                    }
                }
            }
        }
        if (k > 0) {
            // ---- digit 1 (key bits 31..20): from the score kernel's histogram, or this cluster's
            if (!LEAN && !exchange) {
                const uint4* gh = reinterpret_cast<const uint4*>(a.hist + row * H1);
                for (int i = tid; i < H1 / 4; i += NT) reinterpret_cast<uint4*>(s.v.gh)[i] = __ldcg(gh + i);
                __syncthreads();
            } else {
                if (!fused) {
                    for (int i = tid; i < H1; i += NT) s.u.hist[i] = 0u;
                    __syncthreads();
                    for (int p = max(lo, cand_lo) + tid; p < min(hi, cand_hi); p += NT)
                        atomicAdd(&s.u.hist[keys[p - lo] >> 20], 1u);
                }
                __syncthreads();  // the local histogram is complete
                cluster_wait();   // every CTA's copy is zeroed
                // the non-zero bins go to every CTA's copy (a few hundred of the 4096)
                for (int i = tid; i < H1; i += NT) {
                    const uint32_t c = s.u.hist[i];
                    if (c != 0u)
                        for (int r = 0; r < CL; ++r) atomicAdd(cluster.map_shared_rank(&s.v.gh[i], (r + rank) & (CL - 1)), c);
                }
                cluster.sync();  // after it no CTA reads its local histogram again
            }
            find_bin_from_top<H1 / NT>(s.v.gh, (uint32_t)k, s);  // ends with a barrier
            const uint32_t b1 = s.s_bin;
            uint32_t remaining = (uint32_t)k - s.s_above;
            // ---- classification in two phases.  (1) Each lane tests its eight keys against the
            // start of bin b1 (and its positions against the candidate range); the warp queues the
            // lanes with a hit, about a third of them.  (2) Every 32 queued groups, one per lane,
            // are split into kept positions (above bin b1, sinks, window) and candidates (in bin
            // b1), with one packed atomic per warp for the slots of both lists.
            if (tid == 0) s.nsc = 0u;
            __syncthreads();
            const bool inner = lo >= cand_lo && hi <= cand_hi;  // no sink or window position here
            const uint32_t lo_thr = b1 << 20, hi_thr = lo_thr | 0xfffffu;
            static_assert(2 * H2 >= NW * 64, "the warps' queues fit the free digit histograms");
            uint32_t* wq = s.v.w.h2 + warp * 64;  // free until the candidates are broadcast
            int nq = 0;                            // queued groups (uniform over the warp)
            for (int base = 0; base + 256 * warp < n; base += 8 * NT) {  // uniform over the warp
                const int q0 = base + 8 * tid;
                uint32_t m = 0u;
                if (q0 < n) {  // q0 + 8 <= chunk_cap: both loads stay inside the key array
                    const uint4 ka = *reinterpret_cast<const uint4*>(keys + q0);
                    const uint4 kb = *reinterpret_cast<const uint4*>(keys + q0 + 4);
                    const uint32_t kk[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) m |= (uint32_t)(kk[i] >= lo_thr) << i;
                    if (!inner) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int p = lo + q0 + i;
                            m |= (uint32_t)(p < cand_lo || p >= cand_hi) << i;
                        }
                    }
                    m &= (1u << min(n - q0, 8)) - 1u;
                }
                const uint32_t bal = __ballot_sync(0xffffffffu, m != 0u);
                if (m != 0u) wq[nq + __popc(bal & ((1u << lane) - 1u))] = ((uint32_t)q0 << 8) | m;
                nq += __popc(bal);
                if (nq >= 32) {
                    __syncwarp();
                    nq -= 32;
                    classify_group(true, wq[nq + lane], keys, lo, cand_lo, cand_hi, hi_thr, s, lane);
                    __syncwarp();  // the drained slots are refilled
                }
            }
            __syncwarp();
            if (nq > 0) classify_group(lane < nq, lane < nq ? wq[lane] : 0u, keys, lo, cand_lo, cand_hi, hi_thr, s, lane);
            __syncthreads();
            const int n_s0 = (int)(s.nsc & 0xffffu), n_c0 = (int)(s.nsc >> 16);
            // the positions kept so far (above bin b1, sinks and window: all but the few ties at the
            // k-th key) are final.  Their pages are looked up now and their rows pulled into L2 while
            // the candidates are exchanged and the last two digits found, so that the row traffic
            // overlaps the rest of the selection (one-pass list path only)
            static_assert(CAP_S == 2 * NT, "two early list entries per thread");
            n_early = (a.q != nullptr && !has_sel) ? min(n_s0, CAP_S) : 0;
            uint32_t e_pos[2];
            int32_t e_pg[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int i = tid + j * NT;
                e_pos[j] = i < n_early ? s.list[i] : 0u;
                e_pg[j] = (i < n_early && (int)e_pos[j] != t_new)
                              ? __ldg(a.bt + (int64_t)b * a.max_blocks + (e_pos[j] >> 4))
                              : 0;
            }
            // ---- every CTA's candidates (key bits 19..0) go to its slots in every CTA; the
            // target's local histogram is no longer read (see the cluster barrier above)
            {
                const int nc = min(n_c0, CAP_C);
                for (int r0 = 0; r0 < CL; ++r0) {
                    SXSmem* d = cluster.map_shared_rank(&s, (r0 + rank) & (CL - 1));
                    for (int i = tid; i < nc; i += NT)
                        d->u.cand[rank * CAP_C + i] = (uint32_t)(s.v.w.cl[i] >> 32) & 0xfffffu;
                    if (tid == 0) d->ncand[rank] = (uint32_t)n_c0;
                }
            }
            // the fast path's digit histograms and tie counts start from zero
            for (int i = tid; i < H2; i += NT) {
                s.v.w.h2[i] = 0u;
                s.v.w.h2b[i] = 0u;
            }
            if (tid < CL) s.eqr[tid] = 0u;
            if (tid == 0) {
                s.n_s = n_s0;
                s.n_c = n_c0;
                s.nsm = 0u;
            }
            cluster_arrive();  // the broadcast is released; the early rows go out meanwhile
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int i = tid + j * NT;
                if (i < n_early) {
                    const uint32_t r = row_of(a, b, gkv, (int)e_pos[j], t_new, e_pg[j]);
                    s.list[i] = r;
                    if (r < ROW_NEW) {
                        prefetch_row_l2(a.k16 + (int64_t)r * D);
                        prefetch_row_l2(a.v16 + (int64_t)r * D);
                    }
                }
            }
            cluster_wait();
            if (has_hist && rank == 0)  // read by all: clear it for the next layer
                for (int i = tid; i < H1; i += NT) a.hist[row * H1 + i] = 0u;
            bool ovf_c = false;
            for (int r = 0; r < CL; ++r) ovf_c |= s.ncand[r] > (uint32_t)CAP_C;
            if (!ovf_c) {
                // ---- fast path: every CTA finishes the selection over all candidates; slot j
                // of this thread holds rank j's candidate number tid
                uint32_t cr[CL], vm = 0u;
#pragma unroll
                for (int j = 0; j < CL; ++j) {
                    const bool v = (uint32_t)tid < s.ncand[j];
                    cr[j] = v ? s.u.cand[j * CAP_C + tid] : 0u;
                    vm |= (uint32_t)v << j;
                }
#pragma unroll
                for (int j = 0; j < CL; ++j)
                    if ((vm >> j) & 1u) atomicAdd(&s.v.w.h2[cr[j] >> 10], 1u);
                __syncthreads();
                find_bin_from_top<H2 / NT>(s.v.w.h2, remaining, s);
                remaining -= s.s_above;
                const uint32_t d2 = s.s_bin;
                // the candidates sharing digit 2 (usually a few) go to a short list: digit 3 << 3 |
                // owner rank; up to 32 of them one warp finds digit 3 and the per-rank ties at it
#pragma unroll
                for (int j = 0; j < CL; ++j) {
                    if (((vm >> j) & 1u) && (cr[j] >> 10) == d2) {
                        const uint32_t i = atomicAdd(&s.nsm, 1u);
                        if (i < 32u) s.sml[i] = ((cr[j] & (H2 - 1)) << 3) | (uint32_t)j;
                    }
                }
                if (tid == 0) s.bc_cut = 0x7fffffff;
                __syncthreads();
                const uint32_t nsm = s.nsm;
                uint32_t d3;
                if (nsm <= 32u) {
                    if (warp == 0) {
                        const bool valid = (uint32_t)lane < nsm;
                        const uint32_t e = valid ? s.sml[lane] : 0u;
                        const uint32_t v = e >> 3, own = e & (CL - 1);
                        uint32_t gt = 0, eq = 0;
                        for (uint32_t i = 0; i < nsm; ++i) {
                            const uint32_t vi = __shfl_sync(0xffffffffu, v, i);
                            gt += vi > v;
                            eq += vi == v;
                        }
                        // the digit whose run holds the remaining-th largest: above it gt, with it eq
                        const uint32_t hit = __ballot_sync(0xffffffffu, valid && gt < remaining && remaining <= gt + eq);
                        const int src = __ffs(hit) - 1;  // hit != 0: remaining <= nsm entries
                        const uint32_t dv = __shfl_sync(0xffffffffu, v, src), above = __shfl_sync(0xffffffffu, gt, src);
#pragma unroll
                        for (int r = 0; r < CL; ++r) {
                            const uint32_t c = __popc(__ballot_sync(0xffffffffu, valid && v == dv && own == (uint32_t)r));
                            if (lane == 0) s.eqr[r] = c;
                        }
                        if (lane == 0) {
                            s.s_bin = dv;
                            s.s_above = above;
                        }
                    }
                    __syncthreads();
                    remaining -= s.s_above;
                    d3 = s.s_bin;
                } else {  // many share digit 2 (ties): a third histogram pass
#pragma unroll
                    for (int j = 0; j < CL; ++j)
                        if (((vm >> j) & 1u) && (cr[j] >> 10) == d2) atomicAdd(&s.v.w.h2b[cr[j] & (H2 - 1)], 1u);
                    __syncthreads();
                    find_bin_from_top<H2 / NT>(s.v.w.h2b, remaining, s);
                    remaining -= s.s_above;
                    d3 = s.s_bin;
                    const uint32_t low3 = (d2 << 10) | d3;
#pragma unroll
                    for (int j = 0; j < CL; ++j)
                        if (((vm >> j) & 1u) && cr[j] == low3) atomicAdd(&s.eqr[j], 1u);
                    __syncthreads();
                }
                const uint32_t low = (d2 << 10) | d3;
                kth = (b1 << 20) | low;
                // ties at the k-th key: the `remaining` (>= 1) lowest positions among them are kept.
                // Ranks own ascending position ranges, so this CTA keeps its own lowest
                // remaining - (ties in lower ranks) of them, clamped to [0, its ties]
                uint32_t eq_before = 0;
                for (int r = 0; r < rank; ++r) eq_before += s.eqr[r];
                const uint32_t eq_mine = s.eqr[rank];
                const uint32_t keep_t = remaining > eq_before ? min(remaining - eq_before, eq_mine) : 0u;
                const int nc = min(s.n_c, CAP_C);
                if (keep_t == 0) {
                    cut = -1;
                } else if (keep_t == eq_mine) {
                    cut = 0x7fffffff;
                } else {
                    // the keep_t-th lowest position among this CTA's ties
                    for (int i = tid; i < nc; i += NT) {
                        const unsigned long long c = s.v.w.cl[i];
                        if ((uint32_t)(c >> 32) != kth) continue;
                        const uint32_t p = (uint32_t)c;
                        uint32_t r = 0;
                        for (int i2 = 0; i2 < nc; ++i2) {
                            const unsigned long long c2 = s.v.w.cl[i2];
                            r += (uint32_t)(c2 >> 32) == kth && (uint32_t)c2 < p;
                        }
                        if (r == keep_t - 1) s.bc_cut = (int32_t)p;
                    }
                    __syncthreads();
                    cut = s.bc_cut;
                }
                // the kept candidates of this CTA join its list
                for (int i0 = 0; i0 < nc; i0 += NT) {  // uniform bound
                    const int i = i0 + tid;
                    bool f = false;
                    uint32_t p = 0;
                    if (i < nc) {
                        const unsigned long long c = s.v.w.cl[i];
                        const uint32_t key = (uint32_t)(c >> 32);
                        p = (uint32_t)c;
                        f = key > kth || (key == kth && (int32_t)p <= cut);
                    }
                    warp_append<uint32_t>(f, p, s.list, &s.n_s, CAP_S, lane);
                }
                __syncthreads();
                listed = s.n_s <= CAP_S && !has_sel;
            } else {
                // ---- fallback (many candidates share digit 1, e.g. heavy ties): distributed passes
                if (tid == 0 && rank == 0) kvq_dev_count(a.hdr, KVQ_PATH_RADIX_PASSES);
                uint32_t prefix = b1;
                for (int pass = 0; pass < 2; ++pass) {
                    const int shift = pass == 0 ? 10 : 0;
                    for (int i = tid; i < H2; i += NT) s.v.w.h2[i] = 0u;
                    __syncthreads();
                    for (int p = max(lo, cand_lo) + tid; p < min(hi, cand_hi); p += NT) {
                        const uint32_t key = keys[p - lo];
                        if ((key >> (shift + 10)) == prefix) atomicAdd(&s.v.w.h2[(key >> shift) & (H2 - 1)], 1u);
                    }
                    cluster.sync();
                    uint32_t sums[H2 / NT];
#pragma unroll
                    for (int j = 0; j < H2 / NT; ++j) sums[j] = 0u;
                    for (int r = 0; r < CL; ++r) {
                        const uint32_t* rh = cluster.map_shared_rank(s.v.w.h2, r);
#pragma unroll
                        for (int j = 0; j < H2 / NT; ++j) sums[j] += rh[tid + j * NT];
                    }
                    cluster.sync();
#pragma unroll
                    for (int j = 0; j < H2 / NT; ++j) s.v.w.h2[tid + j * NT] = sums[j];
                    __syncthreads();
                    find_bin_from_top<H2 / NT>(s.v.w.h2, remaining, s);
                    remaining -= s.s_above;
                    prefix = (prefix << 10) | s.s_bin;
                }
                kth = prefix;
                // ties: the cut is the remaining-th lowest position with key == kth over the cluster
                uint32_t my_eq = 0;
                for (int p = max(lo, cand_lo) + tid; p < min(hi, cand_hi); p += NT) my_eq += keys[p - lo] == kth;
                uint32_t eq_cta;
                excl_scan<NT>(my_eq, s.wsum, &eq_cta);
                if (tid == 0) {
                    s.eq_cnt = eq_cta;
                    s.bc_cut = 0x7fffffff;
                }
                cluster.sync();
                uint32_t eq_before = 0, eq_total = 0;
                for (int r = 0; r < CL; ++r) {
                    const uint32_t c = cluster.map_shared_rank(&s, r)->eq_cnt;
                    eq_total += c;
                    if (r < rank) eq_before += c;
                }
                if (remaining == 0) {
                    cut = -1;
                } else if (remaining >= eq_total) {
                    cut = 0x7fffffff;
                } else {
                    // the CTA holding the cut finds it with an ordered pass and tells everyone
                    if (eq_before < remaining && remaining <= eq_before + eq_cta) {
                        const uint32_t want = remaining - eq_before;  // 1-based rank inside this CTA
                        uint32_t cnt = 0;
                        for (int p0 = w_lo; p0 < w_hi; p0 += 32) {
                            const int p = p0 + lane;
                            const bool f = p < w_hi && p >= cand_lo && p < cand_hi && keys[p - lo] == kth;
                            cnt += __popc(__ballot_sync(0xffffffffu, f));
                        }
                        if (lane == 0) s.wtot[warp] = cnt;
                        __syncthreads();
                        uint32_t before = 0;
                        for (int w = 0; w < warp; ++w) before += s.wtot[w];
                        if (before < want && want <= before + cnt) {
                            uint32_t run = before;
                            for (int p0 = w_lo; p0 < w_hi; p0 += 32) {
                                const int p = p0 + lane;
                                const bool f = p < w_hi && p >= cand_lo && p < cand_hi && keys[p - lo] == kth;
                                const uint32_t m = __ballot_sync(0xffffffffu, f);
                                if (run + __popc(m) >= want) {
                                    if (f && run + __popc(m & ((1u << lane) - 1u)) + 1 == want)
                                        for (int r = 0; r < CL; ++r) cluster.map_shared_rank(&s, r)->bc_cut = p;
                                    break;
                                }
                                run += __popc(m);
                            }
                        }
                    }
                    cluster.sync();
                    cut = s.bc_cut;
                }
            }
        }
    }
    // the histogram was not needed (everything kept, or k == 0): clear it for the next layer
    if (has_hist && rank == 0 && (keep_all || k == 0))
        for (int i = tid; i < H1; i += NT) a.hist[row * H1 + i] = 0u;

    const uint32_t* plist;  // kept positions of this CTA
    uint32_t nl;
    if (listed) {
        plist = s.list;
        nl = (uint32_t)s.n_s;
    } else {
        // ---- ordered compaction over the chunk (positions ascending), in place into keys[]
        uint32_t cnt = 0;
        for (int it = 0, p0 = w_lo; p0 < w_hi; ++it, p0 += 32) {
            const int p = p0 + lane;
            bool f = p < w_hi;
            if (f && !keep_all && p >= cand_lo && p < cand_hi) {
                const uint32_t key = keys[p - lo];
                f = key > kth || (key == kth && p <= cut);
            }
            const uint32_t m = __ballot_sync(0xffffffffu, f);
            if (lane == 0) s.v.w.wmask[warp][it] = m;
            cnt += __popc(m);
        }
        if (lane == 0) s.wtot[warp] = cnt;
        __syncthreads();  // every key has been read
        uint32_t base = 0;
        nl = 0;
        for (int w = 0; w < NW; ++w) {
            const uint32_t c = s.wtot[w];
            if (w < warp) base += c;
            nl += c;
        }
        for (int it = 0, p0 = w_lo; p0 < w_hi; ++it, p0 += 32) {
            const uint32_t m = s.v.w.wmask[warp][it];
            if ((m >> lane) & 1u) keys[base + __popc(m & ((1u << lane) - 1u))] = (uint32_t)(p0 + lane);
            base += __popc(m);
        }
        plist = keys;
    }
    if (tid == 0) {
        s.sel_cnt = nl;
        kvq_dev_count(a.hdr, listed ? KVQ_PATH_LISTED : KVQ_PATH_COMPACTED);
    }
    __syncthreads();

    if (has_sel) {
        // the ordered selection: this CTA's positions follow those of the lower ranks
        cluster.sync();
        uint32_t off = 0;
        for (int r = 0; r < rank; ++r) off += cluster.map_shared_rank(&s, r)->sel_cnt;
        int32_t* out = a.sel + row * a.sel_cap;
        bool ovf = false;
        for (int i = tid; i < (int)nl; i += NT) {
            if (off + i < (uint32_t)a.sel_cap) out[off + i] = (int32_t)plist[i];
            else ovf = true;
        }
        if (ovf) kvq_dev_flag(a.hdr, KVQ_DEV_OVERFLOW, b);
        if (rank == 0 && tid == 0 && a.sel_count != nullptr) {
            const int total = keep_all ? T : a.n_sink + a.window + k;
            a.sel_count[row] = min(total, a.sel_cap);
        }
        cluster.sync();  // remote counts read before any CTA moves on or leaves
    }
    if (SEL_ONLY || a.q == nullptr) return;

    // ---- attention over this CTA's kept rows
    const int g = gkv;
    // the newest token (appended by this launch, possibly by another cluster) is read from its source
    const uint16_t* knew_row = a.k_new != nullptr ? a.k_new + ((int64_t)b * a.H + g) * D : nullptr;
    const uint16_t* vnew_row = a.k_new != nullptr ? a.v_new + ((int64_t)b * a.H + g) * D : nullptr;
    uint32_t* rows = const_cast<uint32_t*>(plist);  // positions -> row offsets (in 128-element rows)
    // a short list (the sparse heads') goes to L2 at once; a long one (a dense head keeps a whole
    // chunk, megabytes per CTA) a few batches ahead of its use, so that it does not evict itself
    const bool pf_all = nl <= (uint32_t)PF_ALL_MAX;
    for (int i = (listed ? n_early : 0) + tid; i < (int)nl; i += NT) {
        const int t = (int)plist[i];
        const int32_t page = t == t_new ? 0 : a.bt[(int64_t)b * a.max_blocks + (t >> 4)];
        const uint32_t r = row_of(a, b, g, t, t_new, page);
        rows[i] = r;
        // every kept row goes to L2 now; the batches below then mostly hit L2
        if (pf_all && r < ROW_NEW) {
            prefetch_row_l2(a.k16 + (int64_t)r * D);
            prefetch_row_l2(a.v16 + (int64_t)r * D);
        }
    }
    __syncthreads();
    const int hw = tid >> 4, l16 = tid & 15;
    float qv[8];
    {
        const uint4 raw = *reinterpret_cast<const uint4*>(a.q + row * D + 8 * l16);
        unpack8(raw, qv);
#pragma unroll
        for (int i = 0; i < 8; ++i) qv[i] *= KVQ_SCORE_LOG2_SCALE;
    }
    float m = -INFINITY, l = 0.0f, o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = 0.0f;
    for (int it = 0; it < (int)nl; it += NHW * BATCH) {  // bound uniform over the CTA
        if (!pf_all && l16 < 2 * BATCH) {  // lane: row j = l16 / 2 of this half-warp, K or V
            const int i = it + PF_AHEAD * NHW * BATCH + (l16 >> 1) * NHW + hw;
            const uint32_t r = i < (int)nl ? rows[i] : ROW_NONE;
            if (r < ROW_NEW) prefetch_row_l2(((l16 & 1) ? a.v16 : a.k16) + (int64_t)r * D);
        }
        uint4 kr[BATCH], vr[BATCH];
        bool ok[BATCH];
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
            const int i = it + j * NHW + hw;
            const uint32_t r = i < (int)nl ? rows[i] : ROW_NONE;
            ok[j] = r != ROW_NONE;
            kr[j] = make_uint4(0u, 0u, 0u, 0u);
            vr[j] = make_uint4(0u, 0u, 0u, 0u);
            if (ok[j]) {
                const uint16_t* kp = r == ROW_NEW ? knew_row : a.k16 + (int64_t)r * D;
                const uint16_t* vp = r == ROW_NEW ? vnew_row : a.v16 + (int64_t)r * D;
                kr[j] = __ldg(reinterpret_cast<const uint4*>(kp + 8 * l16));
                vr[j] = __ldg(reinterpret_cast<const uint4*>(vp + 8 * l16));
            }
        }
        float sc[BATCH];
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
            float kf[8];
            unpack8(kr[j], kf);
            float acc = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc = fmaf(qv[i], kf[i], acc);
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            sc[j] = ok[j] ? acc : -INFINITY;
        }
        float mn = m;
#pragma unroll
        for (int j = 0; j < BATCH; ++j) mn = fmaxf(mn, sc[j]);
        if (mn != -INFINITY) {
            const float alpha = exp2f(m - mn);
            m = mn;
            l *= alpha;
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] *= alpha;
#pragma unroll
            for (int j = 0; j < BATCH; ++j) {
                const float p = exp2f(sc[j] - mn);
                l += p;
                float vf[8];
                unpack8(vr[j], vf);
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = fmaf(p, vf[i], o[i]);
            }
        }
    }
    // the two half-warps of a warp merge in registers (lanes l and l ^ 16 hold the same channels)
    {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, 16), l2 = __shfl_xor_sync(0xffffffffu, l, 16);
        const float mm = fmaxf(m, m2);
        const float w1 = mm == -INFINITY ? 0.0f : exp2f(m - mm), w2 = mm == -INFINITY ? 0.0f : exp2f(m2 - mm);
        l = l * w1 + l2 * w2;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = o[i] * w1 + __shfl_xor_sync(0xffffffffu, o[i], 16) * w2;
        m = mm;
    }
    // the union buffer is free again: it holds the warp states
    if (lane < 16) {
        float* r = s.v.scratch + warp * REC;
        if (l16 == 0) {
            r[0] = m;
            r[1] = l;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) r[4 + 8 * l16 + i] = o[i];
    }
    __syncthreads();
    SXSmem* r0 = cluster.map_shared_rank(&s, 0);
    if (tid < D) {
        float M = -INFINITY;
        for (int w = 0; w < NW; ++w) M = fmaxf(M, s.v.scratch[w * REC]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
            for (int w = 0; w < NW; ++w) {
                const float wt = exp2f(s.v.scratch[w * REC] - M);
                L = fmaf(s.v.scratch[w * REC + 1], wt, L);
                O = fmaf(s.v.scratch[w * REC + 4 + tid], wt, O);
            }
        }
        r0->st_o[rank][tid] = O;  // push this CTA's state to rank 0
        if (tid == 0) {
            r0->st_m[rank] = M;
            r0->st_l[rank] = L;
        }
    }
    cluster.sync();  // after it no CTA touches another's shared memory
    if (rank == 0 && tid < D) {
        float M = -INFINITY;
        for (int r = 0; r < CL; ++r) M = fmaxf(M, s.st_m[r]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
            for (int r = 0; r < CL; ++r) {
                const float wt = exp2f(s.st_m[r] - M);
                L = fmaf(s.st_l[r], wt, L);
                O = fmaf(s.st_o[r][tid], wt, O);
            }
        }
        a.out[row * D + tid] = L > 0.0f ? O / L : 0.0f;
    }
}

int launch(const SXArgs& a, int batch, cudaStream_t st) {
    const bool lean = a.kT != nullptr && a.sel == nullptr && a.scores_out == nullptr && a.hist == nullptr &&
                      a.q != nullptr && a.n_crit <= 8;
    const bool sel_only = a.kT == nullptr && a.q == nullptr && a.dense == nullptr;
    auto kernel = lean ? select_attn_kernel<1> : sel_only ? select_attn_kernel<2> : select_attn_kernel<0>;
    const int r = kvq_prepare_kernel((const void*)kernel, (int)smem_bytes(MAX_CHUNK));
    if (r) return r;
    const int chunk_cap = chunk_of(a.max_len);
    const cudaError_t e =
        kvq_launch_pdl(kernel, dim3(CL, a.n_heads, batch), dim3(NT), smem_bytes(chunk_cap), st, a, chunk_cap);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "select kernel launch: %s", cudaGetErrorString(e));
    return KVQ_OK;
}

int check_common(const kvq_seqs* S, const char* fn, int32_t n_heads, int32_t k_fixed, double ratio, int32_t n_sink,
                 int32_t window, const float* scores, int64_t score_stride) {
    int st = kvq_check_seqs(S, fn);
    if (st) return st;
    KVQ_REQUIRE(n_heads > 0, KVQ_ERR_INVALID_ARG, "%s: n_heads", fn);
    KVQ_REQUIRE(n_sink >= 0 && window >= 0, KVQ_ERR_INVALID_ARG, "%s: n_sink/window", fn);
    KVQ_REQUIRE(k_fixed >= 0 || (ratio >= 0.0 && ratio <= 1.0), KVQ_ERR_INVALID_ARG, "%s: ratio", fn);
    KVQ_REQUIRE(scores && score_stride >= S->max_len && score_stride % 4 == 0 && ((uintptr_t)scores & 15u) == 0,
                KVQ_ERR_INVALID_ARG, "%s: scores 16-byte aligned, score_stride >= max_len and a multiple of 4", fn);
    KVQ_REQUIRE(chunk_of(S->max_len) <= MAX_CHUNK, KVQ_ERR_UNSUPPORTED, "%s: max_len %d above %d", fn,
                S->max_len, CL * MAX_CHUNK);
    return KVQ_OK;
}

}  // namespace

extern "C" size_t kv_topk_select_ws(void) { return sizeof(KvqWsHeader); }

extern "C" int kv_topk_select(const kvq_seqs* S, int32_t n_heads, const float* scores, int64_t score_stride,
                              int32_t k_fixed, double ratio, int32_t n_sink, int32_t window, int32_t* sel,
                              int32_t sel_cap, int32_t* sel_count, void* ws, size_t ws_bytes, void* stream) {
    kvq_clear_error();
    int st = check_common(S, "kv_topk_select", n_heads, k_fixed, ratio, n_sink, window, scores, score_stride);
    if (st) return st;
    st = kvq_check_ws(ws, ws_bytes, kv_topk_select_ws(), "kv_topk_select");
    if (st) return st;
    KVQ_REQUIRE(sel && sel_count && sel_cap > 0, KVQ_ERR_INVALID_ARG, "kv_topk_select: sel / sel_count / sel_cap");
    if (S->batch == 0) return KVQ_OK;
    SXArgs a{};
    a.scores = scores;
    a.score_stride = score_stride;
    a.hist = nullptr;
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
    a.q = nullptr;
    st = launch(a, S->batch, kvq_stream(stream));
    if (st) return st;
    return kvq_launch_status("kv_topk_select");
}

extern "C" size_t kv_select_sparse_attn_ws(void) { return sizeof(KvqWsHeader); }

extern "C" int kv_select_sparse_attn(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q,
                                     const float* scores, int64_t score_stride, uint32_t* hist, int32_t k_fixed,
                                     double ratio, int32_t n_sink, int32_t window, int32_t* sel, int32_t sel_cap,
                                     int32_t* sel_count, float* out, void* ws, size_t ws_bytes, void* stream) {
    kvq_clear_error();
    int st = kvq_check_layout(L, "kv_select_sparse_attn", true);
    if (st) return st;
    st = check_common(S, "kv_select_sparse_attn", L->n_q_heads, k_fixed, ratio, n_sink, window, scores,
                      score_stride);
    if (st) return st;
    st = kvq_check_ws(ws, ws_bytes, kv_select_sparse_attn_ws(), "kv_select_sparse_attn");
    if (st) return st;
    KVQ_REQUIRE(P && P->k16 && P->v16 && (((uintptr_t)P->k16 | (uintptr_t)P->v16) & 15u) == 0, KVQ_ERR_INVALID_ARG,
                "kv_select_sparse_attn: pool needs 16-byte aligned k16 and v16");
    KVQ_REQUIRE(q && out && ((uintptr_t)q & 15u) == 0, KVQ_ERR_INVALID_ARG, "kv_select_sparse_attn: q / out");
    KVQ_REQUIRE(sel == nullptr || sel_cap > 0, KVQ_ERR_INVALID_ARG, "kv_select_sparse_attn: sel_cap");
    if (S->batch == 0) return KVQ_OK;
    KVQ_REQUIRE(S->block_table != nullptr, KVQ_ERR_INVALID_ARG, "kv_select_sparse_attn: NULL block table");
    SXArgs a{};
    a.scores = scores;
    a.score_stride = score_stride;
    a.hist = hist;
    a.seq_lens = S->seq_lens;
    a.max_len = S->max_len;
    a.n_heads = L->n_q_heads;
    a.k_fixed = k_fixed;
    a.ratio = ratio;
    a.n_sink = n_sink;
    a.window = window;
    a.sel = sel;
    a.sel_cap = sel_cap;
    a.sel_count = sel_count;
    a.hdr = static_cast<KvqWsHeader*>(ws);
    a.q = q;
    a.k16 = P->k16;
    a.v16 = P->v16;
    a.num_blocks = P->num_blocks;
    a.bt = S->block_table;
    a.max_blocks = S->max_blocks;
    a.H = L->n_kv_heads;
    a.GQ = L->n_q_heads / L->n_kv_heads;
    a.out = out;
    st = launch(a, S->batch, kvq_stream(stream));
    if (st) return st;
    return kvq_launch_status("kv_select_sparse_attn");
}

extern "C" size_t kv_sparse_layer_decode_ws(void) { return sizeof(KvqWsHeader); }

static int layer_decode(const char* fn, const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S,
                        const uint16_t* k_new, const uint16_t* v_new, const uint16_t* q, int32_t n_crit,
                        int32_t k_fixed, double ratio, int32_t n_sink, int32_t window, float* scores,
                        int64_t score_stride, int32_t* sel, int32_t sel_cap, int32_t* sel_count, const int32_t* dense,
                        float* out, void* ws, size_t ws_bytes, void* stream) {
    kvq_clear_error();
    int st = kvq_check_layout(L, fn, true);
    if (st) return st;
    st = kvq_check_seqs(S, fn);
    if (st) return st;
    st = kvq_check_ws(ws, ws_bytes, dense ? kvq_dense_heads_attn_ws(L, S) : kv_sparse_layer_decode_ws(), fn);
    if (st) return st;
    KVQ_REQUIRE(L->bits == 16, KVQ_ERR_INVALID_ARG, "%s: not an fp16 layer", fn);
    KVQ_REQUIRE(P && P->k16 && P->v16 && P->kT && P->k_absmax, KVQ_ERR_INVALID_ARG,
                "%s: pool needs k16, v16, kT and k_absmax", fn);
    KVQ_REQUIRE((((uintptr_t)P->k16 | (uintptr_t)P->v16 | (uintptr_t)P->kT) & 15u) == 0, KVQ_ERR_INVALID_ARG,
                "%s: k16, v16 and kT must be 16-byte aligned", fn);
    KVQ_REQUIRE(P->t_cap % 8 == 0 && P->t_cap >= S->max_len && P->t_cap <= (1 << 24), KVQ_ERR_INVALID_ARG,
                "%s: t_cap must be a multiple of 8, >= max_len and <= 2^24", fn);
    KVQ_REQUIRE(n_crit >= 1 && n_crit <= D, KVQ_ERR_INVALID_ARG, "%s: n_crit %d not in [1, 128]", fn, n_crit);
    KVQ_REQUIRE(n_sink >= 0 && window >= 0, KVQ_ERR_INVALID_ARG, "%s: n_sink / window", fn);
    KVQ_REQUIRE(k_fixed >= 0 || (ratio >= 0.0 && ratio <= 1.0), KVQ_ERR_INVALID_ARG, "%s: ratio", fn);
    KVQ_REQUIRE(chunk_of(S->max_len) <= MAX_CHUNK, KVQ_ERR_UNSUPPORTED, "%s: max_len %d above %d", fn, S->max_len,
                CL * MAX_CHUNK);
    KVQ_REQUIRE(scores == nullptr || score_stride >= S->max_len, KVQ_ERR_INVALID_ARG, "%s: score_stride", fn);
    KVQ_REQUIRE(sel == nullptr || (sel_cap > 0 && sel_count != nullptr), KVQ_ERR_INVALID_ARG, "%s: sel", fn);
    KVQ_REQUIRE(S->batch <= P->max_seqs, KVQ_ERR_INVALID_ARG, "%s: batch exceeds max_seqs", fn);
    if (S->batch == 0) return KVQ_OK;
    KVQ_REQUIRE(k_new && v_new && q && out && S->block_table &&
                    (((uintptr_t)q | (uintptr_t)k_new | (uintptr_t)v_new) & 15u) == 0,
                KVQ_ERR_INVALID_ARG, "%s: NULL k_new / v_new / q / out / block table, or q / k_new / v_new not 16-byte aligned", fn);
    SXArgs a{};
    a.scores = nullptr;
    a.score_stride = scores ? score_stride : 0;
    a.hist = nullptr;
    a.seq_lens = S->seq_lens;
    a.max_len = S->max_len;
    a.n_heads = L->n_q_heads;
    a.k_fixed = k_fixed;
    a.ratio = ratio;
    a.n_sink = n_sink;
    a.window = window;
    a.sel = sel;
    a.sel_cap = sel_cap;
    a.sel_count = sel_count;
    a.hdr = static_cast<KvqWsHeader*>(ws);
    a.q = q;
    a.k16 = P->k16;
    a.v16 = P->v16;
    a.num_blocks = P->num_blocks;
    a.bt = S->block_table;
    a.max_blocks = S->max_blocks;
    a.H = L->n_kv_heads;
    a.GQ = L->n_q_heads / L->n_kv_heads;
    a.out = out;
    a.kT = P->kT;
    a.absmax = P->k_absmax;
    a.t_cap = P->t_cap;
    a.n_crit = n_crit;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k16w = P->k16;
    a.v16w = P->v16;
    a.scores_out = scores;
    a.dense = dense;
    a.dense_elsewhere = dense != nullptr;
    cudaStream_t cs = kvq_stream(stream);
    st = launch(a, S->batch, cs);
    if (st) return st;
    st = kvq_launch_status(fn);
    if (st || dense == nullptr) return st;
    // the dense kv heads: every token, the group's q heads sharing each staged tile (stream-ordered
    // after the first launch, which appended the newest token)
    st = kvq_dense_heads_attn(L, P, S, q, dense, out, ws, cs);
    if (st) return st;
    return kvq_launch_status(fn);
}

extern "C" int kv_sparse_layer_decode(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S,
                                      const uint16_t* k_new, const uint16_t* v_new, const uint16_t* q, int32_t n_crit,
                                      int32_t k_fixed, double ratio, int32_t n_sink, int32_t window, float* scores,
                                      int64_t score_stride, int32_t* sel, int32_t sel_cap, int32_t* sel_count,
                                      float* out, void* ws, size_t ws_bytes, void* stream) {
    return layer_decode("kv_sparse_layer_decode", L, P, S, k_new, v_new, q, n_crit, k_fixed, ratio, n_sink, window,
                        scores, score_stride, sel, sel_cap, sel_count, nullptr, out, ws, ws_bytes, stream);
}

extern "C" size_t kv_mixed_layer_decode_ws(const kvq_layout* L, const kvq_seqs* S) {
    if (kvq_check_layout(L, "kv_mixed_layer_decode_ws", true) || kvq_check_seqs_sizes(S, "kv_mixed_layer_decode_ws"))
        return 0;
    return kvq_dense_heads_attn_ws(L, S);
}

extern "C" int kv_mixed_layer_decode(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S,
                                     const uint16_t* k_new, const uint16_t* v_new, const uint16_t* q, int32_t n_crit,
                                     int32_t k_fixed, double ratio, int32_t n_sink, int32_t window,
                                     const int32_t* dense, int32_t* sel, int32_t sel_cap, int32_t* sel_count,
                                     float* out, void* ws, size_t ws_bytes, void* stream) {
    if (dense == nullptr) {
        kvq_clear_error();
        return kvq_fail(KVQ_ERR_INVALID_ARG, "kv_mixed_layer_decode: NULL dense");
    }
    return layer_decode("kv_mixed_layer_decode", L, P, S, k_new, v_new, q, n_crit, k_fixed, ratio, n_sink, window,
                        nullptr, 0, sel, sel_cap, sel_count, dense, out, ws, ws_bytes, stream);
}
