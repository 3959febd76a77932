// f3 outlier-channel isolation [Meeting §8.2]: per (sequence, kv head) the K channels of largest
// variance over the prompt are kept as fp16 in a side cache; in the quantized main cache their
// codes, scale and zero are 0, so they contribute nothing there.  Attention adds their exact
// contribution (kv_decode_attn_quant_outlier).
#include "kvq_internal.cuh"

namespace {

constexpr int D = KVQ_HEAD_DIM;
constexpr int PG = KVQ_BLOCK_TOKENS;
constexpr int KG = KVQ_K_GROUP_TOKENS;
constexpr int MAX_OUT = 8;
static_assert(KG == 64, "the group index below divides by shifting");

// ---- outlier channels: per-channel variance from exact integer sums
//
// Every finite fp16 value is an integer multiple of 2^-24 of magnitude < 2^40 in those units, so
// S1 = sum_t K_t,c (units 2^-24) and S2 = sum_t K_t,c^2 (units 2^-48) are formed exactly, in any
// order: S1 in int64, S2 in three uint64 parts of the magnitude u = a 2^20 + b (u^2 = a^2 2^40 +
// 2ab 2^20 + b^2; each part sums below 2^63 for T <= 2^22).  The sums kernel adds each CTA's
// partial sums into the workspace with 64-bit atomics (integer addition is associative: the totals
// do not depend on the order); the rank kernel rounds S1 and S2 once each to fp64, forms
// Var = (S2 - S1^2 / T) / T with one rounding per operation, picks the n_out largest (ties -> lower
// channel) and zeroes the workspace again.

constexpr int OC_NT = 256;       // threads per CTA: 16 channel groups of 8 x 16 token lanes
constexpr int OC_CHUNK = 2048;   // tokens per CTA
constexpr int OC_MAX_T = 1 << 22;

// fp16 bits -> the value in units of 2^-24 (exact); finite inputs only
__device__ __forceinline__ int64_t h_units(uint32_t h) {
    const uint32_t e = (h >> 10) & 31u, m = h & 1023u;
    const int64_t mag = e == 0 ? (int64_t)m : (int64_t)(m | 1024u) << (e - 1);
    return (h & 0x8000u) ? -mag : mag;
}

// grid (chunks of 2048 tokens, kv heads); thread: channels 8 cg .. 8 cg + 7 (one 16-byte load per
// token) of tokens t0 + lt + 16 j
__global__ void __launch_bounds__(OC_NT) outlier_sums_kernel(const uint16_t* k, int64_t n_tokens, int64_t stride_t,
                                                             unsigned long long* sums) {
    __shared__ unsigned long long part[OC_NT / 32][4][D];
    const int h = blockIdx.y, tid = threadIdx.x, cg = tid & 15, lt = tid >> 4;
    const int64_t t0 = (int64_t)blockIdx.x * OC_CHUNK;
    const int64_t t1 = min(n_tokens, t0 + OC_CHUNK);
    int64_t s1[8];
    unsigned long long p2[8], p1[8], p0[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s1[i] = 0, p2[i] = p1[i] = p0[i] = 0ull;
    const uint16_t* src = k + (int64_t)h * D + 8 * cg;
    for (int64_t t = t0 + lt; t < t1; t += 16) {
        const uint4 w = *reinterpret_cast<const uint4*>(src + t * stride_t);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t x = h_units((ws[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
            s1[i] += x;
            const uint64_t u = (uint64_t)(x < 0 ? -x : x);
            const uint32_t ua = (uint32_t)(u >> 20), ub = (uint32_t)(u & 0xFFFFFu);
            p2[i] += (unsigned long long)ua * ua;
            p1[i] += 2ull * ((unsigned long long)ua * ub);
            p0[i] += (unsigned long long)ub * ub;
        }
    }
    // the warp's two token lanes (lanes l and l + 16 share cg), then the eight warps
    const int warp = tid >> 5;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        unsigned long long v0 = (unsigned long long)s1[i], v1 = p2[i], v2 = p1[i], v3 = p0[i];
        v0 += __shfl_xor_sync(0xffffffffu, v0, 16);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 16);
        v2 += __shfl_xor_sync(0xffffffffu, v2, 16);
        v3 += __shfl_xor_sync(0xffffffffu, v3, 16);
        if ((tid & 31) < 16) {
            part[warp][0][8 * cg + i] = v0;  // two's complement: wrapping sums stay exact
            part[warp][1][8 * cg + i] = v1;
            part[warp][2][8 * cg + i] = v2;
            part[warp][3][8 * cg + i] = v3;
        }
    }
    __syncthreads();
    unsigned long long* dst = sums + (int64_t)h * 4 * D;
    for (int e = tid; e < 4 * D; e += OC_NT) {
        const int w = e / D, c = e % D;
        unsigned long long v = 0;
#pragma unroll
        for (int l = 0; l < OC_NT / 32; ++l) v += part[l][w][c];
        atomicAdd(dst + w * D + c, v);
    }
}

// hi 2^64 + lo rounded to the nearest fp64 (ties to even): the top 64 bits with a sticky bit for
// the rest, rounded by the 64-bit conversion, then scaled by an exact power of two
__device__ __forceinline__ double u128_to_double(uint64_t hi, uint64_t lo) {
    if (hi == 0) return __ull2double_rn(lo);
    const int n = 64 - __clzll((long long)hi);  // bits of hi, 1 .. 64
    uint64_t m, rest;
    if (n == 64) {
        m = hi;
        rest = lo;
    } else {
        m = (hi << (64 - n)) | (lo >> n);
        rest = lo << (64 - n);
    }
    m |= rest != 0 ? 1ull : 0ull;  // far below the rounding position (bit 10 of m)
    return __dmul_rn(__ull2double_rn(m), __longlong_as_double((long long)(1023 + n) << 52));
}

__global__ void __launch_bounds__(D) outlier_rank_kernel(unsigned long long* sums, int64_t n_tokens, int32_t n_out,
                                                         int32_t* out_ch, double* var_out) {
    __shared__ double var[D];
    __shared__ int flag[D];
    const int h = blockIdx.x, c = threadIdx.x;
    unsigned long long* src = sums + (int64_t)h * 4 * D;
    const int64_t S1 = (int64_t)src[c];
    const uint64_t p2 = src[D + c], p1 = src[2 * D + c], p0 = src[3 * D + c];
    src[c] = src[D + c] = src[2 * D + c] = src[3 * D + c] = 0ull;  // leave the workspace zeroed
    // S2 = p2 2^40 + p1 2^20 + p0 as a 128-bit integer
    uint64_t lo = p2 << 40, hi = p2 >> 24;
    const uint64_t l1 = p1 << 20;
    hi += p1 >> 44;
    lo += l1;
    hi += lo < l1 ? 1u : 0u;
    lo += p0;
    hi += lo < p0 ? 1u : 0u;
    double v = 0.0;
    if (n_tokens > 0) {
        const double s1 = __dmul_rn(__ll2double_rn(S1), 0x1p-24);  // exact scalings
        const double s2 = __dmul_rn(u128_to_double(hi, lo), 0x1p-48);
        const double T = (double)n_tokens;
        v = __ddiv_rn(__dsub_rn(s2, __ddiv_rn(__dmul_rn(s1, s1), T)), T);
    }
    var[c] = v;
    if (var_out) var_out[(int64_t)h * D + c] = v;
    __syncthreads();
    int rank = 0;
    for (int j = 0; j < D; ++j) rank += var[j] > v || (var[j] == v && j < c);
    flag[c] = rank < n_out;
    __syncthreads();
    if (flag[c]) {  // ascending channel order: the chosen channels below c
        int pos = 0;
        for (int j = 0; j < c; ++j) pos += flag[j];
        out_ch[(int64_t)h * n_out + pos] = c;
    }
}

struct IsoArgs {
    uint8_t* k_codes;
    uint32_t* k_sz;
    uint16_t* k_out;
    int64_t num_blocks;
    const int32_t* bt;
    const int32_t* seq_lens;
    int32_t max_blocks;
    int32_t H, bits, n_out;
    const int32_t* out_ch;  // [max_seqs][H][n_out]
    // prefill form: the input rows of tokens t_start .. (seq fixed); decode form: k == NULL, the tail
    const uint16_t* k;
    int64_t stride_t, t_start;
    const uint16_t* k_tail;
    int32_t seq;
    KvqWsHeader* hdr;
};

// Isolates the outlier channels of one complete 64-token group (group index gi of sequence b, kv
// head h): thread i < 64 = token 64 gi + i, whose fp16 key at channel c is src[i * ld + c].
__device__ __forceinline__ void isolate_group(const IsoArgs& a, int b, int h, int gi, const uint16_t* src,
                                              int64_t ld) {
    const int i = threadIdx.x;
    const int32_t* ch = a.out_ch + ((int64_t)b * a.H + h) * a.n_out;
    const int32_t page = a.bt[(int64_t)b * a.max_blocks + 4 * gi + i / PG];
    if (page < 0 || page >= a.num_blocks) {
        kvq_dev_flag(a.hdr, KVQ_DEV_BAD_PAGE, b);
        return;
    }
    const int64_t row = ((int64_t)page * a.H + h) * PG + (i % PG);
    uint32_t* codes = reinterpret_cast<uint32_t*>(a.k_codes + row * (D * a.bits / 8));
    const uint32_t M = (1u << a.bits) - 1u;
    for (int j = 0; j < a.n_out; ++j) {
        const int c = ch[j];
        if (c < 0 || c >= D) {  // not a channel: flagged, nothing isolated
            kvq_dev_flag(a.hdr, KVQ_DEV_BAD_INDEX, b);
            a.k_out[row * a.n_out + j] = 0;
            continue;
        }
        a.k_out[row * a.n_out + j] = src[(int64_t)i * ld + c];
        int w, bit;
        kvq_k_code_pos(c, a.bits, &w, &bit);
        codes[w] &= ~(M << bit);  // this thread owns the token's row
        if (i == 0) {             // the group's (scale, zero) sit with its first page
            const int32_t p0 = a.bt[(int64_t)b * a.max_blocks + 4 * gi];
            a.k_sz[((int64_t)p0 * a.H + h) * D + c] = 0u;
        }
    }
}

// prefill form: grid (groups of the range, H); the group's keys come from the input rows
__global__ void __launch_bounds__(KG) isolate_prefill_kernel(IsoArgs a, int64_t n_full) {
    const int gl = blockIdx.x, h = blockIdx.y;
    if (gl >= n_full) return;
    const int gi = (int)(a.t_start >> 6) + gl;  // t_start / 64 (a multiple of 64, checked on the host)
    const uint16_t* base = a.k + (int64_t)gl * KG * a.stride_t + (int64_t)h * D;
    isolate_group(a, a.seq, h, gi, base, a.stride_t);
}

// decode form: grid (H, batch); a sequence whose newest token completed a group (T % 64 == 0)
// isolates that group from its K tail
__global__ void __launch_bounds__(KG) isolate_append_kernel(IsoArgs a) {
    const int h = blockIdx.x, b = blockIdx.y;
    kvq_pdl_begin();
    const int T = a.seq_lens[b];
    if (T <= 0 || T % KG != 0) return;
    const uint16_t* tail = a.k_tail + ((int64_t)b * a.H + h) * KG * D;
    isolate_group(a, b, h, T / KG - 1, tail, D);
}

int check_iso(const kvq_layout* L, const kvq_pool* P, int32_t n_out, const int32_t* out_ch, uint16_t* k_out,
              const char* fn) {
    int st = kvq_check_layout(L, fn, false);
    if (st) return st;
    const int cb = kvq_code_bits(L);
    KVQ_REQUIRE(cb == 4 || cb == 8, KVQ_ERR_UNSUPPORTED, "%s: isolated outlier channels need 4- or 8-bit codes", fn);
    KVQ_REQUIRE(n_out >= 1 && n_out <= MAX_OUT, KVQ_ERR_INVALID_ARG, "%s: n_out %d not in [1, 8]", fn, n_out);
    KVQ_REQUIRE(P && P->k_codes && P->k_sz && out_ch && k_out, KVQ_ERR_INVALID_ARG, "%s: NULL array", fn);
    return KVQ_OK;
}

IsoArgs iso_args(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, int32_t n_out, const int32_t* out_ch,
                 uint16_t* k_out) {
    IsoArgs a{};
    a.k_codes = P->k_codes;
    a.k_sz = reinterpret_cast<uint32_t*>(P->k_sz);
    a.k_out = k_out;
    a.num_blocks = P->num_blocks;
    a.bt = S->block_table;
    a.seq_lens = S->seq_lens;
    a.max_blocks = S->max_blocks;
    a.H = L->n_kv_heads;
    a.bits = kvq_code_bits(L);
    a.n_out = n_out;
    a.out_ch = out_ch;
    a.k_tail = P->k_tail;
    return a;
}

}  // namespace

extern "C" size_t kv_outlier_channels_ws(const kvq_layout* L) {
    if (kvq_check_layout(L, "kv_outlier_channels_ws", false)) return 0;
    return sizeof(KvqWsHeader) + (size_t)L->n_kv_heads * 4 * D * sizeof(unsigned long long);
}

extern "C" int kv_outlier_channels(const kvq_layout* L, const uint16_t* k, int64_t n_tokens, int64_t stride_t,
                                   int32_t n_out, int32_t* out_ch, double* var, void* ws, size_t ws_bytes,
                                   void* stream) {
    kvq_clear_error();
    const char* fn = "kv_outlier_channels";
    int st = kvq_check_layout(L, fn, false);
    if (st) return st;
    KVQ_REQUIRE(out_ch && n_tokens >= 0 && n_tokens <= OC_MAX_T && (k || n_tokens == 0), KVQ_ERR_INVALID_ARG,
                "%s: NULL k / out_ch, or n_tokens outside [0, 2^22]", fn);
    KVQ_REQUIRE(stride_t >= (int64_t)L->n_kv_heads * D && stride_t % 8 == 0 && ((uintptr_t)k & 15u) == 0,
                KVQ_ERR_INVALID_ARG, "%s: stride_t (>= H_kv * d, a multiple of 8) / k (16-byte aligned)", fn);
    KVQ_REQUIRE(n_out >= 1 && n_out <= MAX_OUT, KVQ_ERR_INVALID_ARG, "%s: n_out %d not in [1, 8]", fn, n_out);
    st = kvq_check_ws(ws, ws_bytes, kv_outlier_channels_ws(L), fn);
    if (st) return st;
    unsigned long long* sums =
        reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + sizeof(KvqWsHeader));
    cudaStream_t s = kvq_stream(stream);
    if (n_tokens > 0) {
        const dim3 grid((unsigned)((n_tokens + OC_CHUNK - 1) / OC_CHUNK), L->n_kv_heads);
        outlier_sums_kernel<<<grid, OC_NT, 0, s>>>(k, n_tokens, stride_t, sums);
    }
    outlier_rank_kernel<<<L->n_kv_heads, D, 0, s>>>(sums, n_tokens, n_out, out_ch, var);
    return kvq_launch_status(fn);
}

extern "C" int kv_outlier_isolate(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, int32_t seq,
                                  int64_t t_start, int64_t n_tokens, const uint16_t* k, int64_t stride_t,
                                  int32_t n_out, const int32_t* out_ch, uint16_t* k_out, void* stream) {
    kvq_clear_error();
    const char* fn = "kv_outlier_isolate";
    int st = check_iso(L, P, n_out, out_ch, k_out, fn);
    if (st) return st;
    st = kvq_check_seqs(S, fn);
    if (st) return st;
    KVQ_REQUIRE(seq >= 0 && seq < S->batch && S->block_table, KVQ_ERR_INVALID_ARG, "%s: seq / block table", fn);
    KVQ_REQUIRE(t_start >= 0 && t_start % KG == 0 && n_tokens >= 0 && k, KVQ_ERR_INVALID_ARG,
                "%s: t_start (a multiple of 64), n_tokens, k", fn);
    KVQ_REQUIRE(t_start + n_tokens <= (int64_t)S->max_blocks * PG, KVQ_ERR_INVALID_ARG, "%s: tokens beyond the table",
                fn);
    KVQ_REQUIRE(stride_t >= (int64_t)L->n_kv_heads * D, KVQ_ERR_INVALID_ARG, "%s: stride_t", fn);
    const int64_t n_full = n_tokens / KG;
    if (n_full == 0) return KVQ_OK;
    IsoArgs a = iso_args(L, P, S, n_out, out_ch, k_out);
    a.k = k;
    a.stride_t = stride_t;
    a.t_start = t_start;
    a.seq = seq;
    isolate_prefill_kernel<<<dim3((unsigned)n_full, L->n_kv_heads), KG, 0, kvq_stream(stream)>>>(a, n_full);
    return kvq_launch_status(fn);
}

extern "C" size_t kv_outlier_append_ws(void) { return sizeof(KvqWsHeader); }

extern "C" int kv_outlier_append(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, int32_t n_out,
                                 const int32_t* out_ch, uint16_t* k_out, void* ws, size_t ws_bytes, void* stream) {
    kvq_clear_error();
    const char* fn = "kv_outlier_append";
    int st = check_iso(L, P, n_out, out_ch, k_out, fn);
    if (st) return st;
    st = kvq_check_seqs(S, fn);
    if (st) return st;
    st = kvq_check_ws(ws, ws_bytes, kv_outlier_append_ws(), fn);
    if (st) return st;
    KVQ_REQUIRE(P->k_tail && S->block_table, KVQ_ERR_INVALID_ARG, "%s: k_tail / block table", fn);
    KVQ_REQUIRE(S->batch <= P->max_seqs, KVQ_ERR_INVALID_ARG, "%s: batch exceeds max_seqs", fn);
    if (S->batch == 0) return KVQ_OK;
    IsoArgs a = iso_args(L, P, S, n_out, out_ch, k_out);
    a.hdr = static_cast<KvqWsHeader*>(ws);
    st = kvq_prepare_kernel((const void*)isolate_append_kernel, 0);
    if (st) return st;
    const cudaError_t e =
        kvq_launch_pdl(isolate_append_kernel, dim3(L->n_kv_heads, S->batch), dim3(KG), 0, kvq_stream(stream), a);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "%s launch: %s", fn, cudaGetErrorString(e));
    return KVQ_OK;
}
