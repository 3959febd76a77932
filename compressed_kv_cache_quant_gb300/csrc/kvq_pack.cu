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
template <int BITS, bool SYM>
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
    if constexpr (SYM) {  // scale = max|x| / L, codes offset by L, zero = -L * scale16
        constexpr int L = (1 << (BITS - 1)) - 1;
        const float scale = __fdiv_rn(fmaxf(fabsf(mn), fabsf(mx)), (float)L);
#pragma unroll
        for (int i = 0; i < 4; ++i) codes[i] = kvq_code_sym(x[i], scale, L);
        if ((lane % lpg) == 0) dst_sz[lane / lpg] = pack_sz(scale, kvq_sym_zero(scale, L));
    } else {
        const float levels = (float)((1 << BITS) - 1);
        const float scale = kvq_scale32(mn, mx, levels);
#pragma unroll
        for (int i = 0; i < 4; ++i) codes[i] = kvq_code(x[i], mn, scale, levels);
        if ((lane % lpg) == 0) dst_sz[lane / lpg] = pack_sz(scale, mn);
    }
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

// Codes without a division.  For scale > 0 the code is rint(fl(d / scale)) with d = fl(x - zero)
// (the quotient can't pass the level count, so the clamp never binds).  v = fma(d, 1/scale,
// 1.5 * 2^23) rounds the product to the nearest integer (ties to even) and leaves it in v's low
// mantissa bits; fr = fma(d, 1/scale, 1.5 * 2^23 - v) is the product's distance to that integer.
// Below 256 the product is within 2^-16 of d / scale and the IEEE quotient within 2^-17, so the
// rounding agrees unless |fr| > 1/2 - 2^-15: those codes are redone with the division.  A word is
// the sum of the v bit patterns shifted to their code offsets; the magic constant's share of that
// sum is a per-word constant, subtracted once.  The pairs (lo, hi) of a word go through packed
// fp32x2 arithmetic, which rounds each lane as the scalar instruction does.
constexpr float PK_MAGIC = 12582912.0f;  // 1.5 * 2^23
constexpr uint32_t PK_MAGIC_BITS = 0x4B400000u;
constexpr uint64_t PK_MAGIC2 = 0x4B4000004B400000ull;
constexpr float PK_NEAR = 0.499969482421875f;  // 1/2 - 2^-15
constexpr int PK_KRS = 68;                     // words per staged K row (rows 4 banks apart)

template <int BITS>
__host__ __device__ constexpr uint32_t pk_word_bias() {
    uint32_t c = 0u;
    for (int sl = 0; sl < 16 / BITS; ++sl) c += (PK_MAGIC_BITS << (sl * BITS)) + (PK_MAGIC_BITS << (sl * BITS + 16));
    return c;
}

// The symmetric V words: the same sums of v patterns, each code then offset by L.
template <int BITS>
__host__ __device__ constexpr uint32_t pk_word_bias_sym() {
    uint32_t c = pk_word_bias<BITS>();
    constexpr uint32_t L = BITS >= 2 ? (1u << (BITS - 1)) - 1u : 0u;
    for (int sl = 0; sl < 16 / BITS; ++sl) c -= (L << (sl * BITS)) + (L << (sl * BITS + 16));
    return c;
}

__device__ __forceinline__ uint64_t pk_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void pk_unpack(uint64_t v, uint32_t& lo, uint32_t& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t pk_sub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t pk_fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Adds the codes of the two fp16 values of `xw` (low half at bit `off`, high half at off + 16);
// mn2 and rcp2 hold (zero, 1/scale) of the two values as fp32 pairs.
__device__ __forceinline__ void pk_acc2(uint32_t xw, uint64_t mn2, uint64_t rcp2, int off, uint32_t& acc, float& far) {
    const __half2 h = *reinterpret_cast<const __half2*>(&xw);
    const uint64_t d2 = pk_sub2(pk_pack(__low2float(h), __high2float(h)), mn2);
    const uint64_t v2 = pk_fma2(d2, rcp2, PK_MAGIC2);
    uint32_t flo, fhi, vlo, vhi;
    pk_unpack(pk_fma2(d2, rcp2, pk_sub2(PK_MAGIC2, v2)), flo, fhi);
    pk_unpack(v2, vlo, vhi);
    far = fmaxf(far, fmaxf(fabsf(__uint_as_float(flo)), fabsf(__uint_as_float(fhi))));
    acc += (vlo << off) + (vhi << (off + 16));
}

// The same code, one value: when its quotient is close to a tie, replaces the fast code in `acc`
// by the one the IEEE division gives.
template <int BITS, bool SYM = false>
__device__ __forceinline__ void pk_fix(float x, float mn, float rcp, float sc, int off, uint32_t& acc) {
    const float d = __fsub_rn(x, mn);
    const float v = __fmaf_rn(d, rcp, PK_MAGIC);
    if (fabsf(__fmaf_rn(d, rcp, __fsub_rn(PK_MAGIC, v))) > PK_NEAR) {
        const uint32_t fast = __float_as_uint(v) - PK_MAGIC_BITS;  // signed code (symmetric: before the offset)
        uint32_t exact;
        if constexpr (SYM) {
            constexpr int L = (1 << (BITS - 1)) - 1;
            exact = kvq_code_sym(x, sc, L) - (uint32_t)L;
        } else {
            exact = kvq_code(x, mn, sc, (float)((1 << BITS) - 1));
        }
        acc += (exact - fast) << off;
    }
}

__device__ __forceinline__ __half2 pk_h2(uint32_t u) {
    __half2 h;
    memcpy(&h, &u, 4);
    return h;
}
__device__ __forceinline__ uint32_t pk_u32(__half2 h) {
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
}

// Channel d of the staged V tile sits at column d ^ 8 * (bit 5 of d): the four 16-channel rows
// a warp reads at once then fall in distinct banks.
__device__ __forceinline__ int pk_vcol(int d) { return d ^ (((d >> 5) & 1) << 3); }

// One thread's share of a (64-token group, kv head) unit: 4 chunks of K rows and 2 of V token
// pairs (16 bytes each); rows past the range read as zeros.
struct PkRegs {
    uint4 k[4], va[2], vb[2];
};

__device__ __forceinline__ void pk_load(const PackArgs& a, int gi, int h, int nv, int tid, PkRegs& r) {
    const int c8 = 8 * (tid & 15), i0 = tid >> 4;
    const uint16_t* ksrc = a.k + ((int64_t)gi * KG + i0) * a.stride_t + (int64_t)h * D + c8;
    const uint16_t* vsrc = a.v + ((int64_t)gi * KG + 2 * i0) * a.stride_t + (int64_t)h * D + c8;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        r.k[k] = i0 + 16 * k < nv ? __ldg(reinterpret_cast<const uint4*>(ksrc + (int64_t)(16 * k) * a.stride_t)) : z;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint16_t* r0 = vsrc + (int64_t)(32 * k) * a.stride_t;
        r.va[k] = 2 * i0 + 32 * k < nv ? __ldg(reinterpret_cast<const uint4*>(r0)) : z;
        r.vb[k] = 2 * i0 + 32 * k + 1 < nv ? __ldg(reinterpret_cast<const uint4*>(r0 + a.stride_t)) : z;
    }
}

// K rows as they are (row stride 68 words); V as token pairs, word (y, d) = tokens 2y, 2y+1 at d.
__device__ __forceinline__ void pk_store(const PkRegs& r, uint32_t* kt, uint32_t* vp, int tid) {
    const int c8 = 8 * (tid & 15), i0 = tid >> 4;
#pragma unroll
    for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4*>(kt + (i0 + 16 * k) * PK_KRS + (c8 >> 1)) = r.k[k];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint4 A = r.va[k], B = r.vb[k];
        uint4 lo, hi;
        lo.x = __byte_perm(A.x, B.x, 0x5410); lo.y = __byte_perm(A.x, B.x, 0x7632);
        lo.z = __byte_perm(A.y, B.y, 0x5410); lo.w = __byte_perm(A.y, B.y, 0x7632);
        hi.x = __byte_perm(A.z, B.z, 0x5410); hi.y = __byte_perm(A.z, B.z, 0x7632);
        hi.z = __byte_perm(A.w, B.w, 0x5410); hi.w = __byte_perm(A.w, B.w, 0x7632);
        uint32_t* row = vp + (i0 + 16 * k) * D;
        *reinterpret_cast<uint4*>(row + pk_vcol(c8)) = lo;
        *reinterpret_cast<uint4*>(row + pk_vcol(c8 + 4)) = hi;
    }
}

__device__ __forceinline__ int pk_valid(const PackArgs& a, int gi) {
    return (int)min((int64_t)KG, a.n_tokens - (int64_t)gi * KG);
}

// One CTA of 8 warps per (64-token group, kv head) of the range.
//   1. K rows staged as-is (word p of a row = channels 2p, 2p+1); V rows staged as token pairs
//      (word (y, d) = tokens 2y, 2y+1 at channel d, the pair order of the page layout).
//   2. Statistics: K per channel (complete groups only), V per token and V group.
//   3. Code words, each built whole by one thread straight from the layout: K word (r, q) of
//      token i holds pairs p = 4m + r, m = q*16/b + slot; V word (8t + x, q) of page j holds
//      channels 16t + 8u + x of token pairs r + 4e, m = 4r + 2e + u.  No atomics.
// A page only partly covered keeps its other tokens' V codes; the keys of an unfinished group go
// to the tail buffer.  An invalid table entry skips its page (for K: the group).
template <int BITS, bool SYMV>
__global__ void __launch_bounds__(256) pack_group_kernel(PackArgs a) {
    constexpr int WPR = 4 * BITS;  // K code words per token row
    constexpr int BW = 64 * BITS;  // V code words per page block
    constexpr int PER = 16 / BITS; // codes per half word
    constexpr uint32_t CM = (1u << BITS) - 1u;
    constexpr float LEV = (float)((1 << BITS) - 1);
    constexpr uint32_t BIAS = pk_word_bias<BITS>();
    extern __shared__ __align__(16) unsigned char pk_smem[];
    uint32_t* kt = reinterpret_cast<uint32_t*>(pk_smem);        // [64][68]
    uint32_t* vp = kt + KG * PK_KRS;                             // [32][128] token pairs
    float4* kst = reinterpret_cast<float4*>(vp + (KG / 2) * D);  // [64] per channel pair
    float4* vst = kst + D / 2;                                   // [32][4] per pair and group
    float* ksc = reinterpret_cast<float*>(vst + (KG / 2) * 4);   // [128]
    float* vsc = ksc + D;                                        // [64][4]
    uint32_t* part = reinterpret_cast<uint32_t*>(vsc + KG * 4);  // [2][4][64] half2 min, max of K
    uint32_t* vmm = part + 2 * 256;                              // [32][4][2] half2 min, max of V
    __shared__ int32_t pages[4];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.G, gsh = __ffs(G) - 1, NGV = D >> gsh;
    const int gi = blockIdx.x, h = blockIdx.y;
    const int64_t t0 = a.t_start + (int64_t)gi * KG;  // a multiple of 64: page aligned
    const int nv = pk_valid(a, gi);
    const int npage = (nv + PG - 1) / PG;
    if (tid < 4) {
        int32_t pg = tid < npage ? a.bt_row[t0 / PG + tid] : -1;
        pages[tid] = pg >= 0 && pg < a.pool.num_blocks ? pg : -1;
    }
    {  // ---- 1. staging
        PkRegs rg;
        pk_load(a, gi, h, nv, tid, rg);
        pk_store(rg, kt, vp, tid);
    }
    __syncthreads();
    const bool full = nv == KG;
    const bool k_ok = full && pages[0] >= 0 && pages[1] >= 0 && pages[2] >= 0 && pages[3] >= 0;
    // ---- 2. statistics
    if (k_ok) {  // K: thread (quarter, pair) over 16 tokens
        const int cp = tid & 63, qq = tid >> 6;
        __half2 mn2 = pk_h2(0x7c007c00u), mx2 = pk_h2(0xfc00fc00u);
#pragma unroll 4
        for (int i = 16 * qq; i < 16 * qq + 16; ++i) {
            const __half2 x2 = pk_h2(kt[i * PK_KRS + cp]);
            mn2 = __hmin2(mn2, x2);
            mx2 = __hmax2(mx2, x2);
        }
        part[qq * 64 + cp] = pk_u32(mn2);
        part[256 + qq * 64 + cp] = pk_u32(mx2);
    }
    {  // V: warp w takes token pairs w + 8k (k < 4), lane = 4 channels; pairs past the range are zeros
        __half2 mn2[4], mx2[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 w4 = *reinterpret_cast<const uint4*>(vp + (warp + 8 * k) * D + pk_vcol(4 * lane));
            mn2[k] = __hmin2(__hmin2(pk_h2(w4.x), pk_h2(w4.y)), __hmin2(pk_h2(w4.z), pk_h2(w4.w)));
            mx2[k] = __hmax2(__hmax2(pk_h2(w4.x), pk_h2(w4.y)), __hmax2(pk_h2(w4.z), pk_h2(w4.w)));
        }
        for (int o = 1; o < (G >> 2); o <<= 1) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mn2[k] = __hmin2(mn2[k], pk_h2(__shfl_xor_sync(0xffffffffu, pk_u32(mn2[k]), o)));
                mx2[k] = __hmax2(mx2[k], pk_h2(__shfl_xor_sync(0xffffffffu, pk_u32(mx2[k]), o)));
            }
        }
        if ((lane & ((G >> 2) - 1)) == 0) {  // one lane per group: min and max of the pair
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                vmm[((warp + 8 * k) * 4 + (lane >> (gsh - 2))) * 2] = pk_u32(mn2[k]);
                vmm[((warp + 8 * k) * 4 + (lane >> (gsh - 2))) * 2 + 1] = pk_u32(mx2[k]);
            }
        }
    }
    __syncthreads();
    // scale, zero and 1/scale: thread e < 128 finishes K channel e, the others a V (token, group)
    for (int e = tid; e < D + KG * NGV; e += 256) {
        float mn, mx;
        if (e < D) {
            if (!k_ok) continue;
            const int cp = e >> 1;
            __half2 m2 = pk_h2(part[cp]), x2 = pk_h2(part[256 + cp]);
#pragma unroll
            for (int qq = 1; qq < 4; ++qq) {
                m2 = __hmin2(m2, pk_h2(part[qq * 64 + cp]));
                x2 = __hmax2(x2, pk_h2(part[256 + qq * 64 + cp]));
            }
            mn = (e & 1) ? __high2float(m2) : __low2float(m2);
            mx = (e & 1) ? __high2float(x2) : __low2float(x2);
        } else {
            const int tg = e - D, tok = tg >> (7 - gsh), g = tg & (NGV - 1);
            const uint32_t* mm = vmm + ((tok >> 1) * 4 + g) * 2;
            const __half2 m2 = pk_h2(mm[0]), x2 = pk_h2(mm[1]);
            mn = (tok & 1) ? __high2float(m2) : __low2float(m2);
            mx = (tok & 1) ? __high2float(x2) : __low2float(x2);
        }
        float sc = kvq_scale32(mn, mx, LEV);
        float zs = mn;  // the zero the code words subtract (symmetric V: none)
        if (SYMV && e >= D) {
            sc = __fdiv_rn(fmaxf(fabsf(mn), fabsf(mx)), (float)((1 << (BITS - 1)) - 1));
            zs = 0.0f;
        }
        const float rcp = sc > 0.0f ? 1.0f / sc : 0.0f;
        if (e < D) {
            float* ks4 = reinterpret_cast<float*>(kst + (e >> 1));  // {zero lo, zero hi, 1/sc lo, 1/sc hi}
            ks4[e & 1] = mn;
            ks4[2 + (e & 1)] = rcp;
            ksc[e] = sc;
            a.pool.k_sz[((int64_t)pages[0] * a.H + h) * D + e] = pack_sz(sc, mn);
        } else {
            const int tg = e - D, tok = tg >> (7 - gsh), g = tg & (NGV - 1);
            float* vs4 = reinterpret_cast<float*>(vst + (tok >> 1) * 4 + g);  // {zero even, zero odd, 1/sc ..}
            vs4[tok & 1] = zs;
            vs4[2 + (tok & 1)] = rcp;
            vsc[tok * 4 + g] = sc;
            const int32_t pj = pages[tok / PG];
            const float zst = SYMV ? kvq_sym_zero(sc, (1 << (BITS - 1)) - 1) : mn;
            if (tok < nv && pj >= 0)
                a.pool.v_sz[(((int64_t)pj * a.H + h) * PG + tok % PG) * NGV + g] = pack_sz(sc, zst);
        }
    }
    if (!full) {  // the unfinished group: its keys go to the tail buffer (rows t mod 64 = i)
        uint4* tail = reinterpret_cast<uint4*>(a.pool.k_tail + (((int64_t)a.seq * a.H + h) * KG) * D);
        for (int u = tid; u < nv * 16; u += 256)
            tail[u] = reinterpret_cast<const uint4*>(kt)[(u >> 4) * (PK_KRS / 4) + (u & 15)];
    }
    __syncthreads();
    // ---- 3. code words: K words (r, q) of token 8w + lane/4, V words (8t + x, q) of page w mod 4
    if (k_ok) {
        const int r = lane & 3, i = 8 * warp + (lane >> 2);
        const uint32_t* row = kt + i * PK_KRS + r;
        const ulonglong2* ks = reinterpret_cast<const ulonglong2*>(kst) + r;
        uint32_t* dst = reinterpret_cast<uint32_t*>(a.pool.k_codes) +
                        (((int64_t)pages[i / PG] * a.H + h) * PG + (i % PG)) * WPR + r * BITS;
#pragma unroll
        for (int q = 0; q < BITS; ++q) {
            uint32_t acc = 0u;
            float far = 0.0f;
#pragma unroll
            for (int sl = 0; sl < PER; ++sl) {
                const int p4 = 4 * (q * PER + sl);
                const ulonglong2 st = ks[p4];
                pk_acc2(row[p4], st.x, st.y, sl * BITS, acc, far);
            }
            acc -= BIAS;
            if (far > PK_NEAR) {
#pragma unroll 1
                for (int sl = 0; sl < PER; ++sl) {
                    const int p4 = 4 * (q * PER + sl), c = 2 * (p4 + r);
                    const __half2 x2 = pk_h2(row[p4]);
                    const float4 st = kst[p4 + r];
                    pk_fix<BITS>(__low2float(x2), st.x, st.z, ksc[c], sl * BITS, acc);
                    pk_fix<BITS>(__high2float(x2), st.y, st.w, ksc[c + 1], sl * BITS + 16, acc);
                }
            }
            dst[q] = acc;
        }
    }
    {
        const int x = lane & 7, j = warp & 3, t = 4 * (warp >> 2) + (lane >> 3);
        const int32_t pg = j < npage ? pages[j] : -1;
        if (pg >= 0) {
            const uint32_t* v0 = vp + 8 * j * D + pk_vcol(16 * t + x);      // channel 16t + x
            const uint32_t* v1 = vp + 8 * j * D + pk_vcol(16 * t + 8 + x);  // channel 16t + 8 + x
            const int g = (16 * t) >> gsh;
            const float4* vs = vst + 8 * j * 4 + g;
            uint32_t* dst = reinterpret_cast<uint32_t*>(a.pool.v_codes) + ((int64_t)pg * a.H + h) * BW +
                            (8 * t + x) * BITS;
#pragma unroll
            for (int q = 0; q < BITS; ++q) {
                uint32_t acc = 0u;
                float far = 0.0f;
#pragma unroll
                for (int sl = 0; sl < PER; ++sl) {
                    const int m = q * PER + sl, yl = (m >> 2) + 4 * ((m >> 1) & 1);
                    const ulonglong2 st = reinterpret_cast<const ulonglong2*>(vs)[yl * 4];
                    pk_acc2(((m & 1) ? v1 : v0)[yl * D], st.x, st.y, sl * BITS, acc, far);
                }
                acc -= SYMV ? pk_word_bias_sym<BITS>() : BIAS;
                if (far > PK_NEAR) {
#pragma unroll 1
                    for (int sl = 0; sl < PER; ++sl) {
                        const int m = q * PER + sl, yl = (m >> 2) + 4 * ((m >> 1) & 1), tok = 16 * j + 2 * yl;
                        const __half2 x2 = pk_h2(((m & 1) ? v1 : v0)[yl * D]);
                        const float4 st = vs[yl * 4];
                        pk_fix<BITS, SYMV>(__low2float(x2), st.x, st.z, vsc[tok * 4 + g], sl * BITS, acc);
                        pk_fix<BITS, SYMV>(__high2float(x2), st.y, st.w, vsc[(tok + 1) * 4 + g], sl * BITS + 16,
                                           acc);
                    }
                }
                if (PG * (j + 1) > nv) {  // partly covered page: keep the codes of later tokens
                    uint32_t keep = 0u;
#pragma unroll
                    for (int sl = 0; sl < PER; ++sl) {
                        const int m = q * PER + sl, tok = PG * j + 2 * ((m >> 2) + 4 * ((m >> 1) & 1));
                        if (tok >= nv) keep |= CM << (sl * BITS);
                        if (tok + 1 >= nv) keep |= CM << (sl * BITS + 16);
                    }
                    dst[q] = (dst[q] & keep) | (acc & ~keep);
                } else {
                    dst[q] = acc;
                }
            }
        }
    }
}

constexpr size_t pack_group_smem() {
    return (size_t)KG * PK_KRS * 4 + (size_t)(KG / 2) * D * 4 + (size_t)(D / 2) * 16 + (size_t)(KG / 2) * 4 * 16 +
           (size_t)D * 4 + (size_t)KG * 4 * 4 + 2 * 256 * 4 + (size_t)(KG / 2) * 4 * 2 * 4;
}

// fp16 layer: one CTA of 128 threads per (64-token tile, head).
__global__ void __launch_bounds__(128) pack_fp16_kernel(PackArgs a) {
    const int tile = blockIdx.x;
    const int h = blockIdx.y;
    const int c = threadIdx.x;
    const int64_t i0 = (int64_t)tile * KG;
    const int n = (int)((a.n_tokens - i0) < KG ? (a.n_tokens - i0) : KG);
    float amax = 0.0f;
    const bool has_kT = a.pool.kT != nullptr;  // a layer that is never scored has no channel-major copy
    uint16_t* kT_row = has_kT ? a.pool.kT + (((int64_t)a.seq * a.H + h) * D + c) * a.pool.t_cap : nullptr;
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
        if ((i & 7) == 7 && has_kT) {
            // t - 7 is a multiple of 8 because t_start and the tile start are multiples of 64
            *reinterpret_cast<uint4*>(kT_row + (t - 7)) = *reinterpret_cast<const uint4*>(buf);
        }
    }
    if (!has_kT) return;
    const int rem = n & 7;
    for (int r = 0; r < rem; ++r) kT_row[a.t_start + i0 + (n - rem) + r] = buf[r];
    atomicMax(reinterpret_cast<int*>(a.pool.k_absmax + ((int64_t)a.seq * a.H + h) * D + c), __float_as_int(amax));
}

// fp16 x4 (two f16x2 words) -> E4M3 x4, round to nearest even, finite values saturate at +-448
__device__ __forceinline__ uint32_t e4m3x4(uint32_t lo, uint32_t hi) {
    uint32_t r;
    asm("{\n.reg .b16 a, b;\ncvt.rn.satfinite.e4m3x2.f16x2 a, %1;\ncvt.rn.satfinite.e4m3x2.f16x2 b, %2;\n"
        "mov.b32 %0, {a, b};\n}"
        : "=r"(r) : "r"(lo), "r"(hi));
    return r;
}

// FP8 E4M3 layer: 16 threads per token row (8 values each), 16 rows per CTA; K and V rows cast
// to E4M3 bytes at the row's page slot.
__global__ void __launch_bounds__(256) pack_e4m3_kernel(PackArgs a) {
    const int h = blockIdx.y;
    const int l16 = threadIdx.x & 15;
    const int64_t i = (int64_t)blockIdx.x * 16 + (threadIdx.x >> 4);
    if (i >= a.n_tokens) return;
    const int64_t t = a.t_start + i;
    const int32_t page = a.bt_row[t / PG];
    if (page < 0 || page >= a.pool.num_blocks) return;  // an invalid table entry skips the row
    const int64_t src = i * a.stride_t + (int64_t)h * D + 8 * l16;
    const uint4 kx = *reinterpret_cast<const uint4*>(a.k + src);
    const uint4 vx = *reinterpret_cast<const uint4*>(a.v + src);
    const int64_t dst = (((int64_t)page * a.H + h) * PG + (t % PG)) * D + 8 * l16;
    *reinterpret_cast<uint2*>(a.pool.k_codes + dst) = make_uint2(e4m3x4(kx.x, kx.y), e4m3x4(kx.z, kx.w));
    *reinterpret_cast<uint2*>(a.pool.v_codes + dst) = make_uint2(e4m3x4(vx.x, vx.y), e4m3x4(vx.z, vx.w));
}

template <int BITS, bool SYMV>
int launch_pack_quant(const PackArgs& a, cudaStream_t s) {
    const int64_t n_groups = (a.n_tokens + KG - 1) / KG;
    if (n_groups == 0) return KVQ_OK;
    const int smem = (int)pack_group_smem();
    const int st = kvq_prepare_kernel((const void*)pack_group_kernel<BITS, SYMV>, smem);
    if (st) return st;
    pack_group_kernel<BITS, SYMV><<<dim3((unsigned)n_groups, a.H), 256, smem, s>>>(a);
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

template <int BITS, bool SYMV>
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
        quant_v_token<BITS, SYMV>(vn, a.G, a.pool.v_sz + slot * (D / a.G), c, codes);
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

// FP8 E4M3 layer: the newest token of every (sequence, kv head), 16 threads per row (K and V)
__global__ void __launch_bounds__(32) append_e4m3_kernel(AppendArgs a) {
    const int h = blockIdx.x;
    const int b = blockIdx.y;
    const int l16 = threadIdx.x & 15;
    kvq_pdl_begin();
    const int T = a.seq_lens[b];
    const int64_t p = (int64_t)T - 1;
    if (p < 0) return;
    if (T > a.max_len) {
        if (threadIdx.x == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
        return;
    }
    const int32_t page = page_of(a, b, p / PG);
    if (page < 0) return;
    const bool is_v = threadIdx.x >= 16;
    const uint4 x = *reinterpret_cast<const uint4*>((is_v ? a.v_new : a.k_new) + ((int64_t)b * a.H + h) * D + 8 * l16);
    uint8_t* dst = (is_v ? a.pool.v_codes : a.pool.k_codes) + (((int64_t)page * a.H + h) * PG + (p % PG)) * D + 8 * l16;
    *reinterpret_cast<uint2*>(dst) = make_uint2(e4m3x4(x.x, x.y), e4m3x4(x.z, x.w));
}

__global__ void __launch_bounds__(128) append_fp16_kernel(AppendArgs a) {
    const int h = blockIdx.x;
    const int b = blockIdx.y;
    const int c = threadIdx.x;
    kvq_pdl_begin();
    const int T = a.seq_lens[b];
    const int64_t p = (int64_t)T - 1;
    if (p < 0) return;
    if (T > a.max_len || (a.pool.kT != nullptr && p >= a.pool.t_cap)) {
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
    if (a.pool.kT == nullptr) return;  // a layer that is never scored
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
    if (kvq_code_bits(L) == 16) {
        KVQ_REQUIRE(P->k16 && P->v16 && (P->kT == nullptr) == (P->k_absmax == nullptr), KVQ_ERR_INVALID_ARG,
                    "kv_quant_pack: fp16 layer needs k16, v16, and kT with k_absmax or neither");
        KVQ_REQUIRE(P->kT == nullptr || (P->t_cap % 8 == 0 && t_start + n_tokens <= P->t_cap), KVQ_ERR_INVALID_ARG,
                    "kv_quant_pack: t_cap must be a multiple of 8 covering the tokens");
        KVQ_REQUIRE(((uintptr_t)P->kT & 15u) == 0, KVQ_ERR_INVALID_ARG, "kv_quant_pack: kT must be 16-byte aligned");
        const int64_t tiles = (n_tokens + KG - 1) / KG;
        pack_fp16_kernel<<<dim3((unsigned)tiles, H), 128, 0, s>>>(a);
        return kvq_launch_status("kv_quant_pack");
    }
    if (kvq_code_bits(L) == KVQ_BITS_E4M3) {
        KVQ_REQUIRE(P->k_codes && P->v_codes && (((uintptr_t)P->k_codes | (uintptr_t)P->v_codes) & 7u) == 0,
                    KVQ_ERR_INVALID_ARG, "kv_quant_pack: E4M3 layer needs 8-byte aligned k_codes and v_codes");
        KVQ_REQUIRE(((uintptr_t)k & 15u) == 0 && ((uintptr_t)v & 15u) == 0 && stride_t % 8 == 0, KVQ_ERR_INVALID_ARG,
                    "kv_quant_pack: E4M3 layer needs 16-byte aligned k, v rows (stride_t % 8 == 0)");
        if (n_tokens == 0) return KVQ_OK;
        pack_e4m3_kernel<<<dim3((unsigned)((n_tokens + 15) / 16), H), 256, 0, s>>>(a);
        return kvq_launch_status("kv_quant_pack");
    }
    KVQ_REQUIRE(P->k_codes && P->v_codes && P->k_sz && P->v_sz && P->k_tail, KVQ_ERR_INVALID_ARG,
                "kv_quant_pack: quantized layer needs k_codes, v_codes, k_sz, v_sz, k_tail");
    KVQ_REQUIRE(((uintptr_t)P->k_codes & 15u) == 0 && ((uintptr_t)P->v_codes & 15u) == 0, KVQ_ERR_INVALID_ARG,
                "kv_quant_pack: code arrays must be 16-byte aligned");
    const bool sym = kvq_v_sym(L);
    switch (kvq_code_bits(L)) {
        case 1: return launch_pack_quant<1, false>(a, s);
        case 2: return sym ? launch_pack_quant<2, true>(a, s) : launch_pack_quant<2, false>(a, s);
        case 4: return sym ? launch_pack_quant<4, true>(a, s) : launch_pack_quant<4, false>(a, s);
        default: return sym ? launch_pack_quant<8, true>(a, s) : launch_pack_quant<8, false>(a, s);
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
    if (kvq_code_bits(L) == 16) {
        KVQ_REQUIRE(P->k16 && P->v16 && (P->kT == nullptr) == (P->k_absmax == nullptr), KVQ_ERR_INVALID_ARG,
                    "kv_page_append: fp16 layer needs k16, v16, and kT with k_absmax or neither");
        st = kvq_prepare_kernel((const void*)append_fp16_kernel, 0);
        if (st) return st;
        const cudaError_t e = kvq_launch_pdl(append_fp16_kernel, grid, dim3(128), 0, s, a);
        if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_page_append launch: %s", cudaGetErrorString(e));
        return KVQ_OK;
    }
    if (kvq_code_bits(L) == KVQ_BITS_E4M3) {
        KVQ_REQUIRE(P->k_codes && P->v_codes && (((uintptr_t)P->k_codes | (uintptr_t)P->v_codes) & 7u) == 0,
                    KVQ_ERR_INVALID_ARG, "kv_page_append: E4M3 layer needs 8-byte aligned k_codes and v_codes");
        KVQ_REQUIRE((((uintptr_t)k_new | (uintptr_t)v_new) & 15u) == 0, KVQ_ERR_INVALID_ARG,
                    "kv_page_append: E4M3 layer needs 16-byte aligned k_new and v_new");
        st = kvq_prepare_kernel((const void*)append_e4m3_kernel, 0);
        if (st) return st;
        const cudaError_t e = kvq_launch_pdl(append_e4m3_kernel, grid, dim3(32), 0, s, a);
        if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_page_append launch: %s", cudaGetErrorString(e));
        return KVQ_OK;
    }
    KVQ_REQUIRE(P->k_codes && P->v_codes && P->k_sz && P->v_sz && P->k_tail, KVQ_ERR_INVALID_ARG,
                "kv_page_append: quantized layer needs k_codes, v_codes, k_sz, v_sz, k_tail");
    const int cb = kvq_code_bits(L);
    const bool sym = kvq_v_sym(L);
    void (*fn)(AppendArgs) = cb == 1 ? append_quant_kernel<1, false>
                           : cb == 2 ? (sym ? append_quant_kernel<2, true> : append_quant_kernel<2, false>)
                           : cb == 4 ? (sym ? append_quant_kernel<4, true> : append_quant_kernel<4, false>)
                                     : (sym ? append_quant_kernel<8, true> : append_quant_kernel<8, false>);
    st = kvq_prepare_kernel((const void*)fn, 0);
    if (st) return st;
    const cudaError_t e = kvq_launch_pdl(fn, grid, dim3(128), 0, s, a);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_page_append launch: %s", cudaGetErrorString(e));
    return kvq_launch_status("kv_page_append");
}
