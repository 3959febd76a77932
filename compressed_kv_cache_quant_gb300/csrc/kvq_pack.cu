// a1 kv_quant_pack and a2 kv_page_append: write prompt tokens / one decode
// token into a layer's paged cache.
//
// Quantizer [TailorKV §2.2; OnDevice §3.1]: per group, scale = (max-min)/(2^b-1),
// zero = min, code = clamp(rint((x - zero)/scale), 0, 2^b-1), IEEE fp32 with the
// unrounded scale, scale/zero stored as fp16.  K: per channel over 64 tokens;
// V: per token over G channels.  Paging [KVSurvey §一.1]: 16-token pages found
// through the block table.
#include "kvq_internal.cuh"

namespace {

constexpr int D = KVQ_HEAD_DIM;
constexpr int PG = KVQ_BLOCK_TOKENS;
constexpr int KG = KVQ_K_GROUP_TOKENS;

struct PoolDev {
    uint8_t* k_codes;
    uint8_t* v_codes;
    uint32_t* k_sz;   // (scale, zero) fp16 pairs as one 32-bit word
    uint32_t* v_sz;
    uint16_t* k_tail;
    uint16_t* k16;
    uint16_t* v16;
    uint16_t* kT;
    float* k_absmax;
    int64_t num_blocks;
    int32_t t_cap;
};

PoolDev pool_dev(const kvq_pool* P) {
    PoolDev p;
    p.k_codes = P->k_codes;
    p.v_codes = P->v_codes;
    p.k_sz = reinterpret_cast<uint32_t*>(P->k_sz);
    p.v_sz = reinterpret_cast<uint32_t*>(P->v_sz);
    p.k_tail = P->k_tail;
    p.k16 = P->k16;
    p.v16 = P->v16;
    p.kT = P->kT;
    p.k_absmax = P->k_absmax;
    p.num_blocks = P->num_blocks;
    p.t_cap = P->t_cap;
    return p;
}

__device__ __forceinline__ uint32_t pack_sz(float scale32, float zero) {
    return (uint32_t)kvq_f2h(scale32) | ((uint32_t)kvq_f2h(zero) << 16);
}

// One warp quantizes one V token of 128 channels in groups of G.  Lane l holds channels
// 4l..4l+3 and returns their codes; (scale, zero) of each group goes to dst_sz.
template <int BITS>
__device__ __forceinline__ void quant_v_token(const uint16_t* src, int G, uint32_t* dst_sz, int lane,
                                              uint32_t* codes) {
    const uint2 raw = *reinterpret_cast<const uint2*>(src + 4 * lane);
    float x[4];
    x[0] = kvq_h2f((uint16_t)(raw.x & 0xffffu));
    x[1] = kvq_h2f((uint16_t)(raw.x >> 16));
    x[2] = kvq_h2f((uint16_t)(raw.y & 0xffffu));
    x[3] = kvq_h2f((uint16_t)(raw.y >> 16));
    float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
    float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    const int lpg = G / 4;  // lanes per V group
    for (int o = 1; o < lpg; o <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const float levels = (float)((1 << BITS) - 1);
    const float scale = kvq_scale32(mn, mx, levels);
#pragma unroll
    for (int i = 0; i < 4; ++i) codes[i] = kvq_code(x[i], mn, scale, levels);
    if ((lane % lpg) == 0) dst_sz[lane / lpg] = pack_sz(scale, mn);
}

// Places the four codes of lane l (channels 4l..4l+3) of page token `tok` into a V page block,
// replacing what was there (only this token's bits change).
template <int BITS>
__device__ __forceinline__ void put_v_codes(uint32_t* blk, int tok, int lane, const uint32_t* codes) {
    constexpr uint32_t M = (1u << BITS) - 1u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int w, bit;
        kvq_v_code_pos(tok, 4 * lane + i, BITS, &w, &bit);
        atomicAnd(&blk[w], ~(M << bit));
        if (codes[i]) atomicOr(&blk[w], codes[i] << bit);
    }
}

// Thread c (of 128) quantizes channel c of a 64-token K group read from
// src[i*row_stride + c]; codes are assembled token-major in `rows`
// (64 rows of 4*BITS words, zeroed by the caller) and (scale, zero) of
// channel c is returned in *sz.
template <int BITS>
__device__ __forceinline__ void quant_k_group(const uint16_t* src, int64_t row_stride, int c, uint32_t* rows,
                                              uint32_t* sz) {
    float mn = INFINITY, mx = -INFINITY;
    for (int i = 0; i < KG; ++i) {
        float x = kvq_h2f(src[(int64_t)i * row_stride + c]);
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
    }
    const float levels = (float)((1 << BITS) - 1);
    const float scale = kvq_scale32(mn, mx, levels);
    constexpr int WPR = 4 * BITS;  // 32-bit words per token row
    int word, bit;
    kvq_k_code_pos(c, BITS, &word, &bit);
    for (int i = 0; i < KG; ++i) {
        float x = kvq_h2f(src[(int64_t)i * row_stride + c]);
        uint32_t code = kvq_code(x, mn, scale, levels);
        if (code) atomicOr(&rows[i * WPR + word], code << bit);
    }
    *sz = pack_sz(scale, mn);
}

// Copies 64 assembled K rows to the four pages of their group.
template <int BITS>
__device__ __forceinline__ void store_k_rows(const uint32_t* rows, const int32_t* pages, int H, int h,
                                             uint8_t* k_codes, int tid, int nthreads) {
    constexpr int R = 16 * BITS;            // bytes per row
    constexpr int U4_PER_PAGE = PG * R / 16; // uint4 per page (16 rows)
    const uint4* src = reinterpret_cast<const uint4*>(rows);
    for (int u = tid; u < 4 * U4_PER_PAGE; u += nthreads) {
        const int j = u / U4_PER_PAGE;
        const int r = u % U4_PER_PAGE;
        uint4* dst = reinterpret_cast<uint4*>(k_codes + ((int64_t)pages[j] * H + h) * PG * R);
        dst[r] = src[u];
    }
}

// ------------------------------------------------------------ prefill pack

struct PackArgs {
    PoolDev pool;
    const int32_t* bt_row;  // block table row of the sequence
    int32_t max_blocks;
    int32_t H;
    int32_t G;
    int32_t seq;
    int64_t t_start;
    int64_t n_tokens;
    const uint16_t* k;
    const uint16_t* v;
    int64_t stride_t;
};

// V: one CTA of 4 warps per (page, head) touched by the tokens; the page's block of codes is
// assembled in shared memory (tokens outside the range keep their codes) and written back.
template <int BITS>
__global__ void __launch_bounds__(128) pack_v_kernel(PackArgs a) {
    constexpr int BW = 64 * BITS;  // words per page block
    __shared__ uint32_t blk[BW];
    const int64_t lp = a.t_start / PG + blockIdx.x;  // logical page
    const int h = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t page = a.bt_row[lp];
    if (page < 0 || page >= a.pool.num_blocks) return;  // an invalid table entry skips the page
    uint32_t* gblk = reinterpret_cast<uint32_t*>(a.pool.v_codes) + ((int64_t)page * a.H + h) * BW;
    for (int w = threadIdx.x; w < BW; w += 128) blk[w] = gblk[w];
    __syncthreads();
    for (int tok = warp; tok < PG; tok += 4) {
        const int64_t t = lp * PG + tok;
        if (t < a.t_start || t >= a.t_start + a.n_tokens) continue;  // uniform over the warp
        const int64_t i = t - a.t_start;
        uint32_t codes[4];
        quant_v_token<BITS>(a.v + i * a.stride_t + (int64_t)h * D, a.G,
                            a.pool.v_sz + (((int64_t)page * a.H + h) * PG + tok) * (D / a.G), lane, codes);
        put_v_codes<BITS>(blk, tok, lane, codes);
    }
    __syncthreads();
    for (int w = threadIdx.x; w < BW; w += 128) gblk[w] = blk[w];
}

// K groups: one CTA of 128 threads per (complete 64-token group, head).
template <int BITS>
__global__ void __launch_bounds__(128) pack_k_kernel(PackArgs a) {
    __shared__ __align__(16) uint32_t rows[KG * 4 * BITS];
    __shared__ int32_t pages[4];
    const int gi = blockIdx.x;
    const int h = blockIdx.y;
    const int c = threadIdx.x;
    for (int w = c; w < KG * 4 * BITS; w += 128) rows[w] = 0u;
    const int64_t t0 = a.t_start + (int64_t)gi * KG;
    if (c < 4) pages[c] = a.bt_row[t0 / PG + c];
    __syncthreads();
    for (int j = 0; j < 4; ++j)
        if (pages[j] < 0 || pages[j] >= a.pool.num_blocks) return;  // invalid table entry: skip the group
    uint32_t sz;
    quant_k_group<BITS>(a.k + (int64_t)gi * KG * a.stride_t + (int64_t)h * D, a.stride_t, c, rows, &sz);
    a.pool.k_sz[((int64_t)pages[0] * a.H + h) * D + c] = sz;
    __syncthreads();
    store_k_rows<BITS>(rows, pages, a.H, h, a.pool.k_codes, c, 128);
}

// Keys of the final partial group -> k_tail (rows t mod 64).
__global__ void pack_tail_kernel(PackArgs a, int64_t first_tail, int64_t n_tail) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_tail * a.H * D) return;
    const int c = (int)(idx % D);
    const int h = (int)((idx / D) % a.H);
    const int64_t j = idx / ((int64_t)D * a.H);
    const int64_t t = first_tail + j;     // absolute position
    const int64_t i = t - a.t_start;      // input row
    a.pool.k_tail[(((int64_t)a.seq * a.H + h) * KG + (t % KG)) * D + c] = a.k[i * a.stride_t + (int64_t)h * D + c];
}

// fp16 layer: one CTA of 128 threads per (64-token tile, head).
__global__ void __launch_bounds__(128) pack_fp16_kernel(PackArgs a) {
    const int tile = blockIdx.x;
    const int h = blockIdx.y;
    const int c = threadIdx.x;
    const int64_t i0 = (int64_t)tile * KG;
    const int n = (int)((a.n_tokens - i0) < KG ? (a.n_tokens - i0) : KG);
    float amax = 0.0f;
    uint16_t* kT_row = a.pool.kT + (((int64_t)a.seq * a.H + h) * D + c) * a.pool.t_cap;
    __align__(16) uint16_t buf[8];
    for (int i = 0; i < n; ++i) {
        const int64_t t = a.t_start + i0 + i;
        const int32_t page = a.bt_row[t / PG];
        const uint16_t kx = a.k[(i0 + i) * a.stride_t + (int64_t)h * D + c];
        const uint16_t vx = a.v[(i0 + i) * a.stride_t + (int64_t)h * D + c];
        if (page >= 0 && page < a.pool.num_blocks) {  // an invalid table entry skips the row
            const int64_t off = ((((int64_t)page * a.H + h) * PG) + (t % PG)) * D + c;
            a.pool.k16[off] = kx;
            a.pool.v16[off] = vx;
        }
        amax = fmaxf(amax, fabsf(kvq_h2f(kx)));
        buf[i & 7] = kx;
        if ((i & 7) == 7) {
            // t - 7 is a multiple of 8 because t_start and the tile start are multiples of 64
            *reinterpret_cast<uint4*>(kT_row + (t - 7)) = *reinterpret_cast<const uint4*>(buf);
        }
    }
    const int rem = n & 7;
    for (int r = 0; r < rem; ++r) kT_row[a.t_start + i0 + (n - rem) + r] = buf[r];
    atomicMax(reinterpret_cast<int*>(a.pool.k_absmax + ((int64_t)a.seq * a.H + h) * D + c), __float_as_int(amax));
}

template <int BITS>
int launch_pack_quant(const PackArgs& a, cudaStream_t s) {
    const int64_t n_pages = (a.t_start + a.n_tokens + PG - 1) / PG - a.t_start / PG;
    if (n_pages > 0) pack_v_kernel<BITS><<<dim3((unsigned)n_pages, a.H), 128, 0, s>>>(a);
    const int64_t n_full = a.n_tokens / KG;
    if (n_full > 0) pack_k_kernel<BITS><<<dim3((unsigned)n_full, a.H), 128, 0, s>>>(a);
    const int64_t first_tail = a.t_start + n_full * KG;
    const int64_t n_tail = a.n_tokens - n_full * KG;
    if (n_tail > 0) {
        const int64_t n = n_tail * a.H * D;
        pack_tail_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a, first_tail, n_tail);
    }
    return kvq_launch_status("kv_quant_pack");
}

// ------------------------------------------------------------ decode append

struct AppendArgs {
    PoolDev pool;
    const int32_t* bt;
    const int32_t* seq_lens;
    int32_t max_blocks;
    int32_t max_len;
    int32_t H;
    int32_t G;
    const uint16_t* k_new;
    const uint16_t* v_new;
    KvqWsHeader* hdr;
};

// Returns the page of logical page lp of sequence b, or -1 (flagged) if invalid.
__device__ __forceinline__ int32_t page_of(const AppendArgs& a, int b, int64_t lp) {
    const int32_t p = a.bt[(int64_t)b * a.max_blocks + lp];
    if (p < 0 || p >= a.pool.num_blocks) {
        kvq_dev_flag(a.hdr, KVQ_DEV_BAD_PAGE, b);
        return -1;
    }
    return p;
}

template <int BITS>
__global__ void __launch_bounds__(128) append_quant_kernel(AppendArgs a) {
    __shared__ __align__(16) uint32_t rows[KG * 4 * BITS];
    __shared__ int32_t pages[4];
    __shared__ int ok;
    const int h = blockIdx.x;
    const int b = blockIdx.y;
    const int c = threadIdx.x;
    kvq_pdl_begin();
    const int T = a.seq_lens[b];
    const int64_t p = (int64_t)T - 1;
    if (p < 0) return;
    if (T > a.max_len) {
        if (c == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
        return;
    }
    const int32_t page = page_of(a, b, p / PG);
    if (page < 0) return;
    const uint16_t* kn = a.k_new + ((int64_t)b * a.H + h) * D;
    const uint16_t* vn = a.v_new + ((int64_t)b * a.H + h) * D;
    if (c < 32) {
        const int64_t slot = ((int64_t)page * a.H + h) * PG + (p % PG);
        uint32_t codes[4];
        quant_v_token<BITS>(vn, a.G, a.pool.v_sz + slot * (D / a.G), c, codes);
        put_v_codes<BITS>(reinterpret_cast<uint32_t*>(a.pool.v_codes) + ((int64_t)page * a.H + h) * 64 * BITS,
                          (int)(p % PG), c, codes);
    }
    uint16_t* tail = a.pool.k_tail + ((int64_t)b * a.H + h) * KG * D;
    tail[(p % KG) * D + c] = kn[c];
    if ((p % KG) != KG - 1) return;
    // The token completed a 64-token group: quantize it into its four pages.
    for (int w = c; w < KG * 4 * BITS; w += 128) rows[w] = 0u;
    if (c == 0) ok = 1;
    __syncthreads();
    if (c < 4) {
        const int32_t pg = page_of(a, b, p / PG - 3 + c);
        pages[c] = pg;
        if (pg < 0) ok = 0;
    }
    __syncthreads();
    if (!ok) return;
    uint32_t sz;
    quant_k_group<BITS>(tail, D, c, rows, &sz);
    a.pool.k_sz[((int64_t)pages[0] * a.H + h) * D + c] = sz;
    __syncthreads();
    store_k_rows<BITS>(rows, pages, a.H, h, a.pool.k_codes, c, 128);
}

__global__ void __launch_bounds__(128) append_fp16_kernel(AppendArgs a) {
    const int h = blockIdx.x;
    const int b = blockIdx.y;
    const int c = threadIdx.x;
    kvq_pdl_begin();
    const int T = a.seq_lens[b];
    const int64_t p = (int64_t)T - 1;
    if (p < 0) return;
    if (T > a.max_len || p >= a.pool.t_cap) {
        if (c == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
        return;
    }
    const int32_t page = page_of(a, b, p / PG);
    if (page < 0) return;
    const uint16_t kx = a.k_new[((int64_t)b * a.H + h) * D + c];
    const uint16_t vx = a.v_new[((int64_t)b * a.H + h) * D + c];
    const int64_t off = (((int64_t)page * a.H + h) * PG + (p % PG)) * D + c;
    a.pool.k16[off] = kx;
    a.pool.v16[off] = vx;
    a.pool.kT[(((int64_t)b * a.H + h) * D + c) * a.pool.t_cap + p] = kx;
    float* am = a.pool.k_absmax + ((int64_t)b * a.H + h) * D + c;
    *am = fmaxf(*am, fabsf(kvq_h2f(kx)));
}

}  // namespace

// ------------------------------------------------------------ ABI

extern "C" int kv_quant_pack(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, int32_t seq,
                             int64_t t_start, int64_t n_tokens, const uint16_t* k, const uint16_t* v,
                             int64_t stride_t, void* stream) {
    kvq_clear_error();
    int st = kvq_check_layout(L, "kv_quant_pack", false);
    if (st) return st;
    st = kvq_check_seqs(S, "kv_quant_pack");
    if (st) return st;
    KVQ_REQUIRE(P != nullptr, KVQ_ERR_INVALID_ARG, "kv_quant_pack: NULL pool");
    KVQ_REQUIRE(seq >= 0 && seq < S->batch && seq < P->max_seqs, KVQ_ERR_INVALID_ARG, "kv_quant_pack: seq %d", seq);
    KVQ_REQUIRE(S->block_table != nullptr, KVQ_ERR_INVALID_ARG, "kv_quant_pack: NULL block table");
    KVQ_REQUIRE(t_start >= 0 && t_start % KG == 0, KVQ_ERR_INVALID_ARG,
                "kv_quant_pack: t_start must be a non-negative multiple of 64");
    KVQ_REQUIRE(n_tokens >= 0, KVQ_ERR_INVALID_ARG, "kv_quant_pack: n_tokens < 0");
    KVQ_REQUIRE(t_start + n_tokens <= (int64_t)S->max_blocks * PG, KVQ_ERR_INVALID_ARG,
                "kv_quant_pack: tokens beyond the block table");
    if (n_tokens == 0) return KVQ_OK;
    const int H = L->n_kv_heads;
    KVQ_REQUIRE(k && v, KVQ_ERR_INVALID_ARG, "kv_quant_pack: NULL k/v");
    KVQ_REQUIRE(((uintptr_t)k & 15u) == 0 && ((uintptr_t)v & 15u) == 0, KVQ_ERR_INVALID_ARG,
                "kv_quant_pack: k/v must be 16-byte aligned");
    KVQ_REQUIRE(stride_t >= (int64_t)H * D && stride_t % 8 == 0, KVQ_ERR_INVALID_ARG,
                "kv_quant_pack: stride_t must be >= H_kv*d and a multiple of 8");
    PackArgs a;
    a.pool = pool_dev(P);
    a.bt_row = S->block_table + (int64_t)seq * S->max_blocks;
    a.max_blocks = S->max_blocks;
    a.H = H;
    a.G = L->v_group_dims;
    a.seq = seq;
    a.t_start = t_start;
    a.n_tokens = n_tokens;
    a.k = k;
    a.v = v;
    a.stride_t = stride_t;
    cudaStream_t s = kvq_stream(stream);
    if (L->bits == 16) {
        KVQ_REQUIRE(P->k16 && P->v16 && P->kT && P->k_absmax, KVQ_ERR_INVALID_ARG,
                    "kv_quant_pack: fp16 layer needs k16, v16, kT, k_absmax");
        KVQ_REQUIRE(P->t_cap % 8 == 0 && t_start + n_tokens <= P->t_cap, KVQ_ERR_INVALID_ARG,
                    "kv_quant_pack: t_cap must be a multiple of 8 covering the tokens");
        KVQ_REQUIRE(((uintptr_t)P->kT & 15u) == 0, KVQ_ERR_INVALID_ARG, "kv_quant_pack: kT must be 16-byte aligned");
        const int64_t tiles = (n_tokens + KG - 1) / KG;
        pack_fp16_kernel<<<dim3((unsigned)tiles, H), 128, 0, s>>>(a);
        return kvq_launch_status("kv_quant_pack");
    }
    KVQ_REQUIRE(P->k_codes && P->v_codes && P->k_sz && P->v_sz && P->k_tail, KVQ_ERR_INVALID_ARG,
                "kv_quant_pack: quantized layer needs k_codes, v_codes, k_sz, v_sz, k_tail");
    KVQ_REQUIRE(((uintptr_t)P->k_codes & 15u) == 0 && ((uintptr_t)P->v_codes & 15u) == 0, KVQ_ERR_INVALID_ARG,
                "kv_quant_pack: code arrays must be 16-byte aligned");
    switch (L->bits) {
        case 1: return launch_pack_quant<1>(a, s);
        case 2: return launch_pack_quant<2>(a, s);
        case 4: return launch_pack_quant<4>(a, s);
        default: return launch_pack_quant<8>(a, s);
    }
}

extern "C" size_t kv_page_append_ws(void) { return sizeof(KvqWsHeader); }

extern "C" int kv_page_append(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* k_new,
                              const uint16_t* v_new, void* ws, size_t ws_bytes, void* stream) {
    kvq_clear_error();
    int st = kvq_check_layout(L, "kv_page_append", false);
    if (st) return st;
    st = kvq_check_seqs(S, "kv_page_append");
    if (st) return st;
    st = kvq_check_ws(ws, ws_bytes, kv_page_append_ws(), "kv_page_append");
    if (st) return st;
    KVQ_REQUIRE(P != nullptr && S->block_table != nullptr, KVQ_ERR_INVALID_ARG, "kv_page_append: NULL pool/table");
    KVQ_REQUIRE(S->batch <= P->max_seqs, KVQ_ERR_INVALID_ARG, "kv_page_append: batch exceeds max_seqs");
    if (S->batch == 0) return KVQ_OK;
    KVQ_REQUIRE(k_new && v_new, KVQ_ERR_INVALID_ARG, "kv_page_append: NULL k_new/v_new");
    KVQ_REQUIRE(((uintptr_t)v_new & 7u) == 0, KVQ_ERR_INVALID_ARG, "kv_page_append: v_new must be 8-byte aligned");
    AppendArgs a;
    a.pool = pool_dev(P);
    a.bt = S->block_table;
    a.seq_lens = S->seq_lens;
    a.max_blocks = S->max_blocks;
    a.max_len = S->max_len;
    a.H = L->n_kv_heads;
    a.G = L->v_group_dims;
    a.k_new = k_new;
    a.v_new = v_new;
    a.hdr = static_cast<KvqWsHeader*>(ws);
    cudaStream_t s = kvq_stream(stream);
    dim3 grid(a.H, S->batch);
    if (L->bits == 16) {
        KVQ_REQUIRE(P->k16 && P->v16 && P->kT && P->k_absmax, KVQ_ERR_INVALID_ARG,
                    "kv_page_append: fp16 layer needs k16, v16, kT, k_absmax");
        st = kvq_prepare_kernel((const void*)append_fp16_kernel, 0);
        if (st) return st;
        const cudaError_t e = kvq_launch_pdl(append_fp16_kernel, grid, dim3(128), 0, s, a);
        if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_page_append launch: %s", cudaGetErrorString(e));
        return KVQ_OK;
    }
    KVQ_REQUIRE(P->k_codes && P->v_codes && P->k_sz && P->v_sz && P->k_tail, KVQ_ERR_INVALID_ARG,
                "kv_page_append: quantized layer needs k_codes, v_codes, k_sz, v_sz, k_tail");
    const void* fn = L->bits == 1 ? (const void*)append_quant_kernel<1>
                   : L->bits == 2 ? (const void*)append_quant_kernel<2>
                   : L->bits == 4 ? (const void*)append_quant_kernel<4> : (const void*)append_quant_kernel<8>;
    st = kvq_prepare_kernel(fn, 0);
    if (st) return st;
    cudaError_t e;
    switch (L->bits) {
        case 1: e = kvq_launch_pdl(append_quant_kernel<1>, grid, dim3(128), 0, s, a); break;
        case 2: e = kvq_launch_pdl(append_quant_kernel<2>, grid, dim3(128), 0, s, a); break;
        case 4: e = kvq_launch_pdl(append_quant_kernel<4>, grid, dim3(128), 0, s, a); break;
        default: e = kvq_launch_pdl(append_quant_kernel<8>, grid, dim3(128), 0, s, a); break;
    }
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_page_append launch: %s", cudaGetErrorString(e));
    return kvq_launch_status("kv_page_append");
}
