// f1: block-granular selection -- the block pruning of the meeting article ("长上下文会议大模型推理KV
// 缓存稀疏化与量化联合压缩", §8.1 item 1): rank fixed-size token blocks by the mean of their
// approximate scores and keep the best blocks whole, so that the attention that follows reads
// contiguous runs of rows instead of scattered ones.
//
//   1. block_imp_kernel: importance of every block = mean of the scores of its candidate tokens
//      (n_sink <= t < T - window), an fp32 sum in ascending t divided by the count in fp32;
//      -inf for a block without candidates.
//   2. block_pick_kernel, one CTA per row: the n kept blocks by (importance desc, block asc) --
//      a radix select of the n-th largest order-preserving key in shared memory (four 8-bit
//      digits, most significant first), the blocks above it and, of those equal to it, the
//      lowest-numbered ones -- then the sinks, the kept blocks' tokens and the window as
//      ascending ids.
#include "kvq_internal.cuh"

namespace {

struct BlockImpArgs {
    const float* scores;
    int64_t score_stride;
    const int32_t* seq_lens;
    int32_t max_len;
    int32_t n_heads, n_sink, window, block;
    float* imp;  // [batch][n_heads][imp_stride]
    int64_t imp_stride;
    KvqWsHeader* hdr;
};

__device__ __forceinline__ int clamp_len(int T, int max_len, KvqWsHeader* hdr, int b, bool report) {
    if (T < 0 || T > max_len) {
        if (report) kvq_dev_flag(hdr, KVQ_DEV_BAD_LENGTH, b);
        return T < 0 ? 0 : max_len;
    }
    return T;
}

// Warp w of a CTA owns 32 consecutive blocks, lane l block 32 w + l.  The blocks' tokens pass
// through a shared-memory tile 64 tokens at a time, loaded with coalesced reads; each lane then
// adds its own block's candidate scores in ascending t (fp32).
constexpr int BI_NT = 128, BI_CH = 64;

__global__ void __launch_bounds__(BI_NT) block_imp_kernel(BlockImpArgs a) {
    __shared__ float tile[BI_NT / 32][32][BI_CH + 1];
    const int h = blockIdx.y, b = blockIdx.z, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool first = h == 0 && blockIdx.x == 0 && threadIdx.x == 0;
    const int T = clamp_len(a.seq_lens[b], a.max_len, a.hdr, b, first);
    const int B = a.block, nb = (T + B - 1) / B;
    const int j0 = blockIdx.x * BI_NT + 32 * warp, j = j0 + lane;
    if (j0 >= nb) return;  // uniform over the warp
    const float* s = a.scores + ((int64_t)b * a.n_heads + h) * a.score_stride;
    const int lo = max(j * B, a.n_sink), hi = min((j + 1) * B, T - a.window);
    float acc = 0.0f;
    float(*tl)[BI_CH + 1] = tile[warp];
    for (int c0 = 0; c0 < B; c0 += BI_CH) {
        const int cl = min(BI_CH, B - c0);
#pragma unroll
        for (int i0 = 0; i0 < 32; i0 += 16) {  // 32 loads in flight per lane
            float v[16][2];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int64_t t0 = (int64_t)(j0 + i0 + i) * B + c0;
                v[i][0] = lane < cl && t0 + lane < T ? s[t0 + lane] : 0.0f;
                v[i][1] = lane + 32 < cl && t0 + lane + 32 < T ? s[t0 + lane + 32] : 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                tl[i0 + i][lane] = v[i][0];
                tl[i0 + i][lane + 32] = v[i][1];
            }
        }
        __syncwarp();
        if (j < nb) {
            const int u0 = max(lo - (j * B + c0), 0), u1 = min(hi - (j * B + c0), cl);
            for (int u = u0; u < u1; ++u) acc = __fadd_rn(acc, tl[lane][u]);
        }
        __syncwarp();
    }
    if (j < nb)
        a.imp[((int64_t)b * a.n_heads + h) * a.imp_stride + j] =
            lo < hi ? __fdiv_rn(acc, (float)(hi - lo)) : -INFINITY;
}

struct PickArgs {
    const float* imp;  // [batch][n_heads][imp_stride]
    int64_t imp_stride;
    const int32_t* seq_lens;
    int32_t max_len;
    int32_t n_heads, n_sink, window, block;
    int32_t n_keep_fixed;
    double ratio;
    int32_t* sel;  // [batch][n_heads][sel_cap]
    int32_t sel_cap;
    int32_t* sel_count;
    KvqWsHeader* hdr;
};

constexpr int BP_NT = 1024;
constexpr int BP_MAX_NB = 24576;  // keys of a row in shared memory (96 KB)

// Exclusive scan of one value per thread over the CTA; *total gets the sum.
__device__ __forceinline__ int cta_excl_scan(int v, int* wsum, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < BP_NT / 32 ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < BP_NT / 32) wsum[lane] = w;  // inclusive warp prefix
    }
    __syncthreads();
    const int before = (warp > 0 ? wsum[warp - 1] : 0) + x - v;
    *total = wsum[BP_NT / 32 - 1];
    __syncthreads();  // wsum is reused by the next call
    return before;
}

// Row (b, h).  Output: [0, ns) with ns = min(n_sink, T); the kept blocks' tokens in [ns, wl);
// the window [wl, T) with wl = max(T - window, ns): disjoint parts, ascending.  Thread i owns the
// blocks [i seg, (i + 1) seg) in the two scans (ties among equal keys, output positions).
__global__ void __launch_bounds__(BP_NT) block_pick_kernel(PickArgs a) {
    extern __shared__ uint32_t key[];  // [nb] order-preserving keys of the importances
    __shared__ uint32_t hist[256];
    __shared__ int wsum[BP_NT / 32];
    __shared__ uint32_t s_prefix;
    __shared__ int s_rank;
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int T = clamp_len(a.seq_lens[b], a.max_len, a.hdr, b, h == 0 && tid == 0);
    const int B = a.block, nb = (T + B - 1) / B;
    const int64_t row = (int64_t)b * a.n_heads + h;
    const float* ir = a.imp + row * a.imp_stride;
    int n = a.n_keep_fixed >= 0 ? a.n_keep_fixed : (int)floor(a.ratio * (double)nb);
    n = min(n, nb);
    for (int j = tid; j < nb; j += BP_NT) key[j] = kvq_float_key(ir[j]);
    // the n-th largest key K* (prefix) and how many keys equal to it are kept (rank)
    uint32_t prefix = 0u, mask = 0u;
    int rank = n;
    const bool partial = n > 0 && n < nb;  // uniform over the CTA
    if (partial) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += BP_NT) hist[i] = 0u;
            __syncthreads();
            for (int j = tid; j < nb; j += BP_NT) {
                const uint32_t k = key[j];
                if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (tid < 32) {  // lane l takes bins 255 - 8l down to 248 - 8l
                uint32_t c[8], sum = 0u;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    c[u] = hist[255 - 8 * tid - u];
                    sum += c[u];
                }
                uint32_t x = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
                    if (tid >= o) x += y;
                }
                uint32_t acc = x - sum;  // keys in the bins above this lane's
                if (acc < (uint32_t)rank && (uint32_t)rank <= x) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if ((uint32_t)rank <= acc + c[u]) {
                            s_prefix = prefix | ((uint32_t)(255 - 8 * tid - u) << shift);
                            s_rank = rank - (int)acc;
                            break;
                        }
                        acc += c[u];
                    }
                }
            }
            __syncthreads();
            prefix = s_prefix;
            rank = s_rank;
            mask |= 255u << shift;
        }
    }
    __syncthreads();  // the keys are complete (also when no digit pass ran)
    const int seg = (nb + BP_NT - 1) / BP_NT, j0 = min(nb, tid * seg), j1 = min(nb, j0 + seg);
    int eqc = 0;
    if (partial)
        for (int j = j0; j < j1; ++j) eqc += key[j] == prefix;
    int eqtot;
    const int eq0 = cta_excl_scan(eqc, wsum, &eqtot);
    const int ns = min(a.n_sink, T), wl = max(T - a.window, ns);
    // kept: every block (n == nb), none (n == 0), or key > K*, or key == K* among the first `rank`
    auto kept = [&](int j, int& eqr) {
        if (!partial) return n > 0;
        const uint32_t k = key[j];
        if (k == prefix) return eqr++ < rank;
        return k > prefix;
    };
    int cnt = 0;
    {
        int eqr = eq0;
        for (int j = j0; j < j1; ++j)
            if (kept(j, eqr)) cnt += max(0, min((j + 1) * B, wl) - max(j * B, ns));
    }
    int ctot;
    int pos = ns + cta_excl_scan(cnt, wsum, &ctot);
    int32_t* out = a.sel + row * a.sel_cap;
    {
        int eqr = eq0;
        for (int j = j0; j < j1; ++j) {
            if (!kept(j, eqr)) continue;
            const int lo = max(j * B, ns), c = max(0, min((j + 1) * B, wl) - lo);
            for (int u = 0; u < c; ++u)
                if (pos + u < a.sel_cap) out[pos + u] = lo + u;
            pos += c;
        }
    }
    const int mid_end = ns + ctot, total = mid_end + (T - wl);
    for (int t = tid; t < ns; t += BP_NT)
        if (t < a.sel_cap) out[t] = t;
    for (int t = wl + tid; t < T; t += BP_NT)
        if (mid_end + (t - wl) < a.sel_cap) out[mid_end + (t - wl)] = t;
    if (tid == 0) {
        if (total > a.sel_cap) kvq_dev_flag(a.hdr, KVQ_DEV_OVERFLOW, b);
        a.sel_count[row] = min(total, a.sel_cap);
    }
}

struct BlockWs {
    size_t off_imp, total;
    int64_t imp_stride;
    int32_t max_nb;
};

BlockWs block_ws(const kvq_seqs* S, int32_t n_heads, int32_t block) {
    BlockWs w{};
    const int64_t B = std::max(S->batch, 1);
    w.max_nb = (std::max(S->max_len, 1) + block - 1) / block;
    w.imp_stride = kvq_round_up((size_t)w.max_nb, 4);
    w.off_imp = kvq_round_up(sizeof(KvqWsHeader), 256);
    w.total = kvq_round_up(w.off_imp + (size_t)B * n_heads * (size_t)w.imp_stride * sizeof(float), 256);
    return w;
}

}  // namespace

extern "C" size_t kv_block_select_ws(const kvq_seqs* S, int32_t n_heads, int32_t block_tokens) {
    if (kvq_check_seqs_sizes(S, "kv_block_select_ws") || n_heads <= 0 || block_tokens <= 0) return 0;
    return block_ws(S, n_heads, block_tokens).total;
}

extern "C" int kv_block_select(const kvq_seqs* S, int32_t n_heads, const float* scores, int64_t score_stride,
                               int32_t n_keep_fixed, double ratio, int32_t n_sink, int32_t window,
                               int32_t block_tokens, int32_t* sel, int32_t sel_cap, int32_t* sel_count, void* ws,
                               size_t ws_bytes, void* stream) {
    kvq_clear_error();
    int st = kvq_check_seqs(S, "kv_block_select");
    if (st) return st;
    KVQ_REQUIRE(n_heads > 0, KVQ_ERR_INVALID_ARG, "kv_block_select: n_heads");
    KVQ_REQUIRE(block_tokens >= 1 && block_tokens <= 4096, KVQ_ERR_INVALID_ARG, "kv_block_select: block_tokens %d",
                block_tokens);
    KVQ_REQUIRE(n_sink >= 0 && window >= 0, KVQ_ERR_INVALID_ARG, "kv_block_select: n_sink/window");
    KVQ_REQUIRE(n_keep_fixed >= 0 || (ratio >= 0.0 && ratio <= 1.0), KVQ_ERR_INVALID_ARG, "kv_block_select: ratio");
    KVQ_REQUIRE(scores && score_stride >= S->max_len, KVQ_ERR_INVALID_ARG, "kv_block_select: scores / score_stride");
    KVQ_REQUIRE(sel && sel_count && sel_cap > 0, KVQ_ERR_INVALID_ARG, "kv_block_select: sel / sel_count / sel_cap");
    const BlockWs w = block_ws(S, n_heads, block_tokens);
    KVQ_REQUIRE(w.max_nb <= BP_MAX_NB, KVQ_ERR_UNSUPPORTED, "kv_block_select: %d blocks per row, at most %d",
                w.max_nb, BP_MAX_NB);
    st = kvq_check_ws(ws, ws_bytes, w.total, "kv_block_select");
    if (st) return st;
    if (S->batch == 0) return KVQ_OK;
    cudaStream_t s = kvq_stream(stream);
    char* base = static_cast<char*>(ws);
    BlockImpArgs ia{};
    ia.scores = scores;
    ia.score_stride = score_stride;
    ia.seq_lens = S->seq_lens;
    ia.max_len = S->max_len;
    ia.n_heads = n_heads;
    ia.n_sink = n_sink;
    ia.window = window;
    ia.block = block_tokens;
    ia.imp = reinterpret_cast<float*>(base + w.off_imp);
    ia.imp_stride = w.imp_stride;
    ia.hdr = static_cast<KvqWsHeader*>(ws);
    st = kvq_prepare_kernel((const void*)block_imp_kernel, 0);
    if (st) return st;
    block_imp_kernel<<<dim3((unsigned)((w.max_nb + BI_NT - 1) / BI_NT), (unsigned)n_heads, (unsigned)S->batch),
                       BI_NT, 0, s>>>(ia);
    st = kvq_launch_status("kv_block_select");
    if (st) return st;
    PickArgs pa{};
    pa.imp = ia.imp;
    pa.imp_stride = w.imp_stride;
    pa.seq_lens = S->seq_lens;
    pa.max_len = S->max_len;
    pa.n_heads = n_heads;
    pa.n_sink = n_sink;
    pa.window = window;
    pa.block = block_tokens;
    pa.n_keep_fixed = n_keep_fixed;
    pa.ratio = ratio;
    pa.sel = sel;
    pa.sel_cap = sel_cap;
    pa.sel_count = sel_count;
    pa.hdr = static_cast<KvqWsHeader*>(ws);
    const int smem = w.max_nb * (int)sizeof(uint32_t);
    st = kvq_prepare_kernel((const void*)block_pick_kernel, BP_MAX_NB * (int)sizeof(uint32_t));
    if (st) return st;
    block_pick_kernel<<<dim3((unsigned)n_heads, (unsigned)S->batch), BP_NT, smem, s>>>(pa);
    return kvq_launch_status("kv_block_select");
}
