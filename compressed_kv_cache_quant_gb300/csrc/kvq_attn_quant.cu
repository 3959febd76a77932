// a3 kv_decode_attn_quant: fused dequant -> q.k/sqrt(d) -> online softmax ->
// p.v over the quantized paged cache [OnDevice §3.2; TailorKV §2.2], with the
// context split across CTAs and the partial softmax states merged by
// log-sum-exp in the last CTA of every (sequence, kv head).
//
// Both contractions run on the tensor cores (mma.sync m16n8k16, fp16 in, fp32
// accumulate), one warp per 64-token group (one K quantization group = four
// 16-token pages).  With K = scale_c * code + zero_c per channel of the group,
//   s_t = sum_c (q_c scale_c) code_t[c] + sum_c q_c zero_c,
// the first term is a [tokens x 128] x [128 x slots] product whose A operand
// is 1 + code / 2^b, made two codes at a time by one shift and one AND/OR into
// the mantissa of fp16 1.0 (the codes are stored in pairs for that,
// kvq_k_code_pos), and whose B operand holds q_c scale_c 2^b (exact in fp32)
// split into two fp16 halves (a hi and a lo column per head, summed
// afterwards); the bias sum_c q_c scale_c 2^b joins the zero-point term.  With V = vscale_t
// code + vzero_t per token and V group,
//   o[d] = sum_t p_t (vscale_t code_t[d] + vzero_t)
// is a [128 x tokens] x [tokens x columns] product whose A operand is the V codes (stored
// channel-major per page, kvq_v_code_pos) made exact fp16 numbers.  When the heads times the V
// groups per token fit the product's eight columns (all but 4 heads with 32-dim V groups), column
// NGV h + j holds fp16(2^8 p_t vscale_t) of head h and V group j (the softmax weights taken as
// 2^8 p, which the normalisation cancels), the zero points join as an fp32 sum of p_t vzero_t per column, and a channel's output is read from its group's column; otherwise
// the A operand is fp16(vscale_t code + vzero_t), one more fp16 FMA per pair, against p_t in fp16
// (column 2h).  The group's codes and scales are staged per warp with cp.async, one
// group ahead.  An unfinished K group reads its keys from the fp16 tail buffer.
#include <algorithm>

#include "kvq_internal.cuh"

namespace {

constexpr int D = KVQ_HEAD_DIM;
constexpr int PG = KVQ_BLOCK_TOKENS;
constexpr int KG = KVQ_K_GROUP_TOKENS;
// warps per CTA: 16 for 1- and 2-bit codes (one CTA per SM); 4-bit codes run in small CTAs
// of 2 warps, several per SM (the measured best on a batch of MHA sequences of differing
// lengths); 8-bit codes, whose staged groups are the largest, in CTAs of 4 warps
template <int BITS>
__host__ __device__ constexpr int nwarp_of() {
    return BITS <= 2 ? 16 : (BITS == 4 ? 2 : 4);
}
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
    int32_t H;       // kv heads of the cache
    int32_t kv_div;  // grid kv groups per kv head (2 when 8 q heads share one: two halves of 4)
    int32_t G;       // V group dims
    const uint16_t* q;
    float* out;
    float* part;
    int32_t* counters;
    KvqWsHeader* hdr;
    int32_t n_splits;
    int32_t cps;     // 64-token groups per split
    // isolated outlier channels (the outlier form of the kernel only): fp16 keys of the packed
    // tokens [num_blocks][H][16][n_out], the channels [batch][H][n_out]
    const uint16_t* k_out = nullptr;
    const int32_t* out_ch = nullptr;
    int32_t n_out = 0;
};

// ---------------------------------------------------------------- small helpers

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// d += A (16x16, row) * B (16x8, col), fp16 operands, fp32 accumulators
__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// byte permute: the 4 bytes of the result chosen from {a, b} by the selector's nibbles
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}
// fp16x2 a * b + c, one rounding per half
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

__device__ __forceinline__ float2 unpack_h2(uint32_t x) {
    return make_float2(kvq_h2f((uint16_t)(x & 0xffffu)), kvq_h2f((uint16_t)(x >> 16)));
}

// The code pair at bit offset POS (< 16) of both halves of w as two fp16 numbers.  The bits are
// moved to offset E < 10 - BITS + 1 of the fp16 mantissa of 1024, giving 1024 + 2^E code
// exactly; one fp16 FMA with 2^-E and -2^(10-E) then gives the code exactly.
template <int BITS, int POS>
__device__ __forceinline__ uint32_t code_pair(uint32_t w) {
    constexpr int X = BITS <= 2 ? 10 : 8;
    constexpr int SH = POS - POS % X;
    constexpr int E = POS - SH;
    static_assert(E + BITS <= 10, "the code fits the fp16 mantissa");
    constexpr uint32_t M = (1u << BITS) - 1u;
    constexpr uint32_t MASK = (M << E) | (M << (16 + E));
    const uint32_t x = ((w >> SH) & MASK) | 0x64006400u;
    constexpr uint32_t SC = (uint32_t)(0x3C00 - (E << 10));                 // 2^-E
    constexpr uint32_t OF = (uint32_t)(0x8000 | ((25 - E) << 10));          // -2^(10-E)
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(SC | (SC << 16)), "r"(OF | (OF << 16)));
    return r;
}

// K B-fragment register for pair m of this lane's column (see kvq_k_code_pos): kw = the
// BITS words of the column in the token row.  The codes go to the top BITS mantissa bits of
// fp16 1.0, giving 1 + code / 2^BITS exactly with one shift and one AND/OR; the 2^BITS factor
// and the bias of 1 are taken up by the A operand and the per-head constant.
template <int BITS, int M>
__device__ __forceinline__ uint32_t k_pair(const uint32_t* kw) {
    constexpr int PER = 16 / BITS;
    constexpr int POS = (M % PER) * BITS;
    constexpr int SH = POS - (10 - BITS);  // right shift (left if negative)
    constexpr uint32_t M1 = ((1u << BITS) - 1u) << (10 - BITS);
    const uint32_t w = kw[M / PER];
    const uint32_t x = SH >= 0 ? (w >> (SH >= 0 ? SH : 0)) : (w << (SH < 0 ? -SH : 0));
    return (x & (M1 | (M1 << 16))) | 0x3C003C00u;
}

// The four V A-fragment registers of column r (pairs m = 4r .. 4r + 3, kvq_v_code_pos) from
// the BITS words of row 8t + x of the page block.
template <int BITS>
__device__ __forceinline__ void v_pairs(const uint32_t* vw, int r, uint32_t* A) {
    if constexpr (BITS == 1) {
        const uint32_t x = vw[0] >> (4 * r);
        A[0] = code_pair<1, 0>(x);
        A[1] = code_pair<1, 1>(x);
        A[2] = code_pair<1, 2>(x);
        A[3] = code_pair<1, 3>(x);
    } else if constexpr (BITS == 2) {
        const uint32_t x = vw[r >> 1] >> (8 * (r & 1));
        A[0] = code_pair<2, 0>(x);
        A[1] = code_pair<2, 2>(x);
        A[2] = code_pair<2, 4>(x);
        A[3] = code_pair<2, 6>(x);
    } else if constexpr (BITS == 4) {
        const uint32_t x = vw[r];
        A[0] = code_pair<4, 0>(x);
        A[1] = code_pair<4, 4>(x);
        A[2] = code_pair<4, 8>(x);
        A[3] = code_pair<4, 12>(x);
    } else {
        const uint32_t x0 = vw[2 * r], x1 = vw[2 * r + 1];
        A[0] = code_pair<8, 0>(x0);
        A[1] = code_pair<8, 8>(x0);
        A[2] = code_pair<8, 0>(x1);
        A[3] = code_pair<8, 8>(x1);
    }
}

// ---------------------------------------------------------------- the kernel

// One warp's staged 64-token group.
template <int BITS>
struct GroupStage {
    uint32_t k[KG * 4 * BITS];   // K token rows (complete groups only)
    uint32_t v[4 * 64 * BITS];   // V page blocks
    uint32_t ksz[D];             // K (scale, zero) per channel
    uint32_t vsz[KG * 4];        // V (scale, zero) per token and V group (at most 4 groups)
};

constexpr int AFR_LD = 36;  // padded row: the lanes' stores of one register row hit distinct banks

template <int BITS, int GQ, int NWARP = nwarp_of<BITS>()>
struct QMSmem {
    float qs[GQ][D];                  // the query heads of the kv group times 2^BITS (fp32)
    float m[NWARP][GQ], l[NWARP][GQ];
    uint32_t afr[NWARP][16][AFR_LD];  // per warp: the scores' A fragments, [register][lane]
    union alignas(16) {               // cp.async writes 16-byte chunks into the stages
        GroupStage<BITS> st[NWARP][2];
        float ro[NWARP][GQ][D];       // per warp: unnormalised outputs, after the last group
    } u;
};

// The outlier form adds, after QMSmem in dynamic shared memory, per warp and stage the fp16
// outlier keys of the group's 64 tokens (token-major, n_out <= 8 per token): 128 n_out bytes each
constexpr int MAX_OUT = 8;
template <int BITS>
__host__ __device__ constexpr size_t ko_bytes(int n_out) {
    return (size_t)nwarp_of<BITS>() * 2 * KG * n_out * sizeof(uint16_t);
}

// Issues the cp.async copies of group gi into st (one warp); pages past the sequence are
// skipped (their tokens are masked), complete groups also bring their K rows and scales.
// Lane i < 4: the block-table entry of page i of group gi (-1 past the sequence), loaded an
// iteration before stage_group needs it.
__device__ __forceinline__ int32_t group_page(const QAttnArgs& a, int b, int gi, int n_pages, int lane) {
    const int lp = 4 * gi + lane;
    return lane < 4 && lp < n_pages ? a.bt[(int64_t)b * a.max_blocks + lp] : -1;
}

template <int BITS, int NGV, bool OUT = false>
__device__ __forceinline__ void stage_group(const QAttnArgs& a, GroupStage<BITS>& st, int b, int gk, int gi,
                                            int n_full, int32_t pg, int lane, uint16_t* ko = nullptr) {
    if (lane < 4 && pg != -1 && (pg < 0 || pg >= a.num_blocks)) {
        kvq_dev_flag(a.hdr, KVQ_DEV_BAD_PAGE, b);
        pg = 0;
    }
    const int32_t P0 = __shfl_sync(0xffffffffu, pg, 0), P1 = __shfl_sync(0xffffffffu, pg, 1);
    const int32_t P2 = __shfl_sync(0xffffffffu, pg, 2), P3 = __shfl_sync(0xffffffffu, pg, 3);
    const bool packed = gi < n_full;
    constexpr int CH = 16 * BITS;  // 16-byte chunks per page of K rows, and per V page block
#pragma unroll
    for (int c0 = 0; c0 < 4 * CH; c0 += 32) {
        const int c = c0 + lane, i = c / CH, r = c % CH;
        const int32_t P = i == 0 ? P0 : i == 1 ? P1 : i == 2 ? P2 : P3;
        if (c >= 4 * CH || P < 0) continue;
        const int64_t off = (((int64_t)P * a.H + gk) * PG) * (16 * BITS) + 16 * r;
        if (packed) cp_async16(st.k + (i * CH + r) * 4, a.k_codes + off);
        cp_async16(st.v + (i * CH + r) * 4, a.v_codes + off);
    }
    if (packed) cp_async16(st.ksz + 4 * lane, a.k_sz + ((int64_t)P0 * a.H + gk) * D + 4 * lane);
    constexpr int VCH = 4 * NGV;  // chunks of V scales per page
#pragma unroll
    for (int c0 = 0; c0 < 4 * VCH; c0 += 32) {
        const int c = c0 + lane, i = c / VCH, r = c % VCH;
        const int32_t P = i == 0 ? P0 : i == 1 ? P1 : i == 2 ? P2 : P3;
        if (c >= 4 * VCH || P < 0) continue;
        cp_async16(st.vsz + i * 16 * NGV + 4 * r, a.v_sz + ((int64_t)P * a.H + gk) * PG * NGV + 4 * r);
    }
    if constexpr (OUT) {  // the packed tokens' outlier keys: 32 n_out bytes per page
        const int nc = 2 * a.n_out;
        if (packed)
            for (int c = lane; c < 4 * nc; c += 32) {
                const int i = (c >= nc) + (c >= 2 * nc) + (c >= 3 * nc), r = c - i * nc;
                const int32_t P = i == 0 ? P0 : i == 1 ? P1 : i == 2 ? P2 : P3;
                if (P < 0) continue;
                cp_async16(ko + i * PG * a.n_out + 8 * r, a.k_out + ((int64_t)P * a.H + gk) * PG * a.n_out + 8 * r);
            }
    }
}

// OUT: the outlier form (isolated outlier channels of the keys, meeting article §8.2): their codes,
// scales and zeros are 0 in the main cache, and their fp16 keys, staged beside the group's codes,
// add sum_j q_(c_j) K_(t, c_j) to the packed tokens' scores.
// (the 4-bit outlier form is held to 168 registers: three 2-warp CTAs' warps per SM sub-partition, so
// that shared memory, not registers, limits it to five CTAs per SM as the plain form)
template <int BITS, int GQ, int NGV, bool OUT = false>  // NGV = 128 / v_group_dims V groups per token
__global__ void __launch_bounds__(32 * nwarp_of<BITS>(), OUT && BITS == 4 ? 6 : 1) qmma_kernel(QAttnArgs a) {
    constexpr int NWARP = nwarp_of<BITS>(), NT = 32 * NWARP;
    static_assert(GQ <= 4, "at most four query heads per grid kv group");
    extern __shared__ __align__(16) unsigned char smraw[];
    QMSmem<BITS, GQ>& S = *reinterpret_cast<QMSmem<BITS, GQ>*>(smraw);
    uint16_t* const ko_base = reinterpret_cast<uint16_t*>(smraw + sizeof(QMSmem<BITS, GQ>));  // OUT only
    __shared__ int is_last;

    const int split = blockIdx.x, gv = blockIdx.y, b = blockIdx.z;
    const int Hv = gridDim.y, Hq = Hv * GQ;
    const int gk = gv / a.kv_div;  // kv head of the codes
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, q4 = lane & 3;  // fragment row group / column pair
    kvq_pdl_begin();
    const int T = a.seq_lens[b];
    if (T > a.max_len || T < 0) {
        if (tid == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
        return;
    }
    const int n_full = T / KG;
    const int n_groups = (T + KG - 1) / KG;
    const int n_pages = (T + PG - 1) / PG;
    const int nsplit_b = (n_groups + a.cps - 1) / a.cps;
    if (n_groups == 0) {  // empty sequence: output 0
        if (split == 0)
            for (int i = tid; i < GQ * D; i += NT) a.out[((int64_t)b * Hq + gv * GQ) * D + i] = 0.0f;
        return;
    }
    if (split >= nsplit_b) return;
    const int g_begin = split * a.cps, g_end = min(n_groups, g_begin + a.cps);

    for (int i = tid; i < GQ * D; i += NT)  // q 2^BITS (exact): the codes enter as 1 + code / 2^BITS
        S.qs[i / D][i % D] = kvq_h2f(a.q[((int64_t)b * Hq + gv * GQ) * D + i]) * (float)(1 << BITS);
    // A-fragment rows of absent heads (fewer than four) stay zero
    for (int i = tid; i < NWARP * 16 * AFR_LD; i += NT) (&S.afr[0][0][0])[i] = 0u;
    __syncthreads();

    float acc[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][i] = 0.0f;
    float mrun = -INFINITY, lrun = 0.0f;
    [[maybe_unused]] const int hs = g8 >> 1;  // the head of this lane's score rows (slot g8 = 2 hs + hi/lo)
    // With GQ NGV <= 8 the value product's eight B columns hold one (head, V group) each: column
    // g8 = NGV h + j, so that the V scales go into B and the codes enter the A operand as they are
    constexpr bool VCOL = GQ * NGV <= 8;
    [[maybe_unused]] const int jn = g8 % NGV;                 // this lane's B column: V group jn
    [[maybe_unused]] const bool vcol = g8 / NGV < GQ;         //   of head g8 / NGV, if present
    [[maybe_unused]] const int vsrc = min(g8 / NGV, GQ - 1);  // (clamped: a lane to read from)
    float zacc = 0.0f;  // sum_t p_t vzero_t of column g8 over this lane's tokens
    // outlier form: the score product gets one more k-step per m-tile whose k slots are the
    // outlier channels j < n_out (k = 2 q4, 2 q4 + 1 in this lane's registers): B column 2h holds
    // q of head h at channel c_j (fp16, exact), A the staged fp16 outlier keys of the tokens
    uint32_t ob0 = 0u;
    bool has0 = false, has1 = false;
    int oj0 = 0, oj1 = 0;       // the lane's two k slots, clamped into the row (branch-free loads)
    uint32_t omask = 0u;        // the halves of the A register that are real slots
    if constexpr (OUT) {
        has0 = 2 * q4 < a.n_out;
        has1 = 2 * q4 + 1 < a.n_out;
        oj0 = min(2 * q4, a.n_out - 1);
        oj1 = min(2 * q4 + 1, a.n_out - 1);
        omask = (has0 ? 0x0000ffffu : 0u) | (has1 ? 0xffff0000u : 0u);
        float qlo = 0.0f, qhi = 0.0f;
        const int32_t* chs = a.out_ch + ((int64_t)b * a.H + gk) * a.n_out;
        const int c0 = has0 ? chs[2 * q4] : 0, c1 = has1 ? chs[2 * q4 + 1] : 0;
        if (c0 < 0 || c0 >= D || c1 < 0 || c1 >= D) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_INDEX, b);
        const int h = g8 >> 1;
        if ((g8 & 1) == 0 && h < GQ) {  // q 2^BITS back to q: exact
            if (has0 && c0 >= 0 && c0 < D) qlo = S.qs[h][c0] * (1.0f / (float)(1 << BITS));
            if (has1 && c1 >= 0 && c1 < D) qhi = S.qs[h][c1] * (1.0f / (float)(1 << BITS));
        }
        ob0 = pack_h2(qlo, qhi);
    }
    auto ko_of = [&](int bf) -> uint16_t* { return OUT ? ko_base + (warp * 2 + bf) * KG * a.n_out : nullptr; };

    int gi = g_begin + warp, buf = 0;
    if (gi < g_end)
        stage_group<BITS, NGV, OUT>(a, S.u.st[warp][0], b, gk, gi, n_full, group_page(a, b, gi, n_pages, lane), lane,
                                    ko_of(0));
    cp_commit();
    int32_t pg_next = group_page(a, b, gi + NWARP, n_pages, lane);
    for (; gi < g_end; gi += NWARP) {
        if (gi + NWARP < g_end)
            stage_group<BITS, NGV, OUT>(a, S.u.st[warp][buf ^ 1], b, gk, gi + NWARP, n_full, pg_next, lane,
                                        ko_of(buf ^ 1));
        cp_commit();
        pg_next = group_page(a, b, gi + 2 * NWARP, n_pages, lane);
        cp_wait<1>();
        __syncwarp();
        const GroupStage<BITS>& st = S.u.st[warp][buf];
        const int t0 = gi * KG;
        const bool packed = gi < n_full;
        [[maybe_unused]] const uint16_t* kob = OUT ? ko_of(buf) + g8 * a.n_out : nullptr;  // outlier keys, row g8

        // ---- A fragments: slot 2h holds fp16(q_h,c scale_c), slot 2h + 1 the fp16 remainder;
        // register 2s + i covers channels 16s + 8i + 2r + {0, 1} of fragment column r
        float c0p[GQ];
#pragma unroll
        for (int h = 0; h < GQ; ++h) c0p[h] = 0.0f;
#pragma unroll
        for (int k = 0; k < 2 * GQ; ++k) {
            const int u = lane + 32 * k;
            const int h = k >> 1, s = (u >> 3) & 7, i = (u >> 2) & 1, r = u & 3;
            const int c = 16 * s + 8 * i + 2 * r;
            const float2 qv = *reinterpret_cast<const float2*>(&S.qs[h][c]);
            // complete group: a_c = q_c scale_c 2^BITS (q, scale fp16: exact in fp32) against the
            // codes' 1 + code / 2^BITS; the unfinished group: a_c = q_c against fp16 keys
            // (the query in shared memory is q 2^BITS: a power of two, exact)
            float a0, a1;
            if (packed) {
                const float2 sz0 = unpack_h2(st.ksz[c]), sz1 = unpack_h2(st.ksz[c + 1]);
                a0 = qv.x * sz0.x;
                a1 = qv.y * sz1.x;
                // zero-point term minus the bias sum_c a_c (hi + lo misses a_c by < 2^-22 |a_c|)
                c0p[h] += fmaf(qv.x, sz0.y, qv.y * sz1.y) * (1.0f / (float)(1 << BITS)) - (a0 + a1);
            } else {
                a0 = qv.x * (1.0f / (float)(1 << BITS));
                a1 = qv.y * (1.0f / (float)(1 << BITS));
            }
            if (!(fabsf(a0) < 32768.0f && fabsf(a1) < 32768.0f)) kvq_dev_flag(a.hdr, KVQ_DEV_RANGE, b);
            const uint32_t hi = pack_h2(a0, a1);
            const float2 hf = unpack_h2(hi);
            const uint32_t lo = pack_h2(a0 - hf.x, a1 - hf.y);
            S.afr[warp][2 * s + i][4 * (2 * h) + r] = hi;
            S.afr[warp][2 * s + i][4 * (2 * h + 1) + r] = lo;
        }
        float c0 = 0.0f;  // of head q4, the head of this lane's scores
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            const float v = kvq_warp_sum(c0p[h]);
            if (q4 == h) c0 = v;
        }
        __syncwarp();
        uint32_t af[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) af[r] = S.afr[warp][r][lane];

        // ---- scores: the A operand is the codes (16 tokens x 16 channels per m-tile and k-step:
        // tokens 16mt + g8 and + 8, channel pairs 2s and 2s + 1 of the lane's column), the B
        // operand the fragments above (slot 2h: hi, 2h + 1: lo of head h); this lane gets
        // head q4 of tokens 16mt + g8 (hi in d0, lo in d1) and 16mt + g8 + 8 (d2, d3)
        float sc[4][2];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (packed) {
                const uint32_t* k0 = st.k + (16 * mt + g8) * (4 * BITS) + q4 * BITS;
                const uint32_t* k1 = k0 + 8 * (4 * BITS);
                uint32_t w0[BITS], w1[BITS];
#pragma unroll
                for (int u = 0; u < BITS; ++u) {
                    w0[u] = k0[u];
                    w1[u] = k1[u];
                }
#define KVQ_KSTEP(S)                                                                                       \
    mma16816(d, k_pair<BITS, 2 * (S)>(w0), k_pair<BITS, 2 * (S)>(w1), k_pair<BITS, 2 * (S) + 1>(w0),       \
             k_pair<BITS, 2 * (S) + 1>(w1), af[2 * (S)], af[2 * (S) + 1])
                KVQ_KSTEP(0);
                KVQ_KSTEP(1);
                KVQ_KSTEP(2);
                KVQ_KSTEP(3);
                KVQ_KSTEP(4);
                KVQ_KSTEP(5);
                KVQ_KSTEP(6);
                KVQ_KSTEP(7);
#undef KVQ_KSTEP
                if constexpr (OUT) {  // the outlier channels of tokens 16mt + g8 (+ 8): exact fp16 keys
                    const uint16_t* kr = kob + 16 * mt * a.n_out;  // row 16mt + g8 of the stage
                    const uint16_t* kr8 = kr + 8 * a.n_out;
                    const uint32_t oa0 = prmt(kr[oj0], kr[oj1], 0x5410u) & omask;
                    const uint32_t oa1 = prmt(kr8[oj0], kr8[oj1], 0x5410u) & omask;
                    mma16816(d, oa0, oa1, 0u, 0u, ob0, 0u);
                }
            } else {
                // the unfinished group: fp16 keys (rows t mod 64 of the tail buffer), q unscaled
                const uint32_t* k0 = reinterpret_cast<const uint32_t*>(
                    a.k_tail + (((int64_t)b * a.H + gk) * KG + 16 * mt + g8) * D + 2 * q4);
                const uint32_t* k1 = k0 + 8 * D / 2;
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma16816(d, k0[8 * s], k1[8 * s], k0[8 * s + 4], k1[8 * s + 4], af[2 * s], af[2 * s + 1]);
            }
            sc[mt][0] = d[0] + d[1];
            sc[mt][1] = d[2] + d[3];
        }
        // ---- online softmax of head q4 (log2 domain) over the group's 64 tokens: eight per lane
        float gm = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = t0 + 16 * mt + g8 + 8 * e;
                sc[mt][e] = t < T ? (sc[mt][e] + c0) * KVQ_SCORE_LOG2_SCALE : -INFINITY;
                gm = fmaxf(gm, sc[mt][e]);
            }
        gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 4));
        gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 8));
        gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 16));
        const float mn = fmaxf(mrun, gm);
        const float alpha = mn == -INFINITY ? 1.0f : exp2f(mrun - mn);
        // with the V scales in B the weights are taken as 2^8 p (l and o scale alike, o / l does
        // not change), so that fp16(2^8 p vscale) stays normal down to p vscale = 2^-22
        const float mp = VCOL ? mn - 8.0f : mn;
        float ls = 0.0f;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float p = mn == -INFINITY ? 0.0f : exp2f(sc[mt][e] - mp);
                sc[mt][e] = p;
                ls += p;
            }
        mrun = mn;
        lrun = fmaf(lrun, alpha, ls);
        if constexpr (VCOL) {
            // accumulator column n = 2 q4 + c is (head n / NGV, V group n % NGV); only the m-tiles
            // of that group are read at the end
            float al0 = alpha, al1 = alpha;
            if constexpr (NGV != 2) {
                al0 = __shfl_sync(0xffffffffu, alpha, min((2 * q4) / NGV, GQ - 1));
                al1 = __shfl_sync(0xffffffffu, alpha, min((2 * q4 + 1) / NGV, GQ - 1));
            }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int j = (mt * NGV) >> 3;  // resolved at compile time
                if (NGV == 1 || (j & 1) == 0) {
                    acc[mt][0] *= al0;
                    acc[mt][2] *= al0;
                }
                if (NGV == 1 || (j & 1) == 1) {
                    acc[mt][1] *= al1;
                    acc[mt][3] *= al1;
                }
            }
            zacc *= __shfl_sync(0xffffffffu, alpha, vsrc);  // column g8's head
        } else {
            // the accumulator columns belong to head q4 too
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                acc[mt][0] *= alpha;
                acc[mt][2] *= alpha;
            }
        }

        if constexpr (VCOL) {
            // ---- values: the A operand is the codes themselves (exact in fp16: the pair at tokens
            // 2q4, 2q4 + 1 and 2q4 + 8, 2q4 + 9 of page ks, channels g8 and g8 + 8 of the m-tile); B
            // column g8 = NGV h + j carries fp16(2^8 p_t vscale_t) of head h and V group j, and the
            // zero points join as sum_t p_t vzero_t per column, in fp32.  The code and zero-point
            // sums are of similar size and opposite sign, so the tensor cores sum one group at a
            // time from zero and the group's sums join the running ones by fp32 additions.
            uint32_t bb[4][2];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                // p of head vsrc at the page's tokens 2q4, 2q4 + 1, 2q4 + 8, 2q4 + 9: token y sits
                // in lane 4 (y mod 8) + vsrc, register e = y / 8 of m-tile ks
                const float p0 = __shfl_sync(0xffffffffu, sc[ks][0], 8 * q4 + vsrc);
                const float p1 = __shfl_sync(0xffffffffu, sc[ks][0], 8 * q4 + 4 + vsrc);
                const float p2 = __shfl_sync(0xffffffffu, sc[ks][1], 8 * q4 + vsrc);
                const float p3 = __shfl_sync(0xffffffffu, sc[ks][1], 8 * q4 + 4 + vsrc);
                const int tb = 16 * ks + 2 * q4;             // the lane's first token in the group
                const int nv = vcol ? T - t0 - tb : 0;       // tokens tb, tb + 1 valid if > 0, > 1; tb + 8, + 9 if > 8, > 9
                const uint32_t* vz = st.vsz + tb * NGV + jn;  // (scale, zero) of V group jn per token
                // masked tokens and absent columns: scale and zero 0 (their staged words may hold anything)
                const float2 u0 = unpack_h2(nv > 0 ? vz[0] : 0u);
                const float2 u1 = unpack_h2(nv > 1 ? vz[NGV] : 0u);
                const float2 u2 = unpack_h2(nv > 8 ? vz[8 * NGV] : 0u);
                const float2 u3 = unpack_h2(nv > 9 ? vz[9 * NGV] : 0u);
                // 2^8 p vscale must stay finite in fp16: |vscale| < 256
                if (!(fmaxf(fmaxf(fabsf(u0.x), fabsf(u1.x)), fmaxf(fabsf(u2.x), fabsf(u3.x))) < 256.0f))
                    kvq_dev_flag(a.hdr, KVQ_DEV_RANGE, b);
                bb[ks][0] = pack_h2(p0 * u0.x, p1 * u1.x);
                bb[ks][1] = pack_h2(p2 * u2.x, p3 * u3.x);
                zacc = fmaf(p0, u0.y, fmaf(p1, u1.y, fmaf(p2, u2.y, fmaf(p3, u3.y, zacc))));
            }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t A[4];
                    v_pairs<BITS>(st.v + ks * 64 * BITS + (8 * mt + g8) * BITS, q4, A);
                    mma16816(d, A[0], A[1], A[2], A[3], bb[ks][0], bb[ks][1]);
                }
                const int j = (mt * NGV) >> 3;  // resolved at compile time: the columns read at the end
                if (NGV == 1 || (j & 1) == 0) {
                    acc[mt][0] += d[0];
                    acc[mt][2] += d[2];
                }
                if (NGV == 1 || (j & 1) == 1) {
                    acc[mt][1] += d[1];
                    acc[mt][3] += d[3];
                }
            }
        } else {
            // ---- values, page by page: the A operand is the dequantized V, fp16(vscale code + vzero)
            // (the codes' pair at tokens 2q4, 2q4 + 1 and 2q4 + 8, 2q4 + 9 of the page, channels g8 and
            // g8 + 8 of the m-tile); the B column g8 = 2h carries fp16(p) of head h, odd columns 0
            const bool even = (g8 & 1) == 0 && hs < GQ;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                // p of head hs at the page's tokens 2q4, 2q4 + 1, 2q4 + 8, 2q4 + 9: token y sits in lane
                // 4 (y mod 8) + hs, register e = y / 8 of m-tile ks
                const float p0 = __shfl_sync(0xffffffffu, sc[ks][0], 8 * q4 + hs);
                const float p1 = __shfl_sync(0xffffffffu, sc[ks][0], 8 * q4 + 4 + hs);
                const float p2 = __shfl_sync(0xffffffffu, sc[ks][1], 8 * q4 + hs);
                const float p3 = __shfl_sync(0xffffffffu, sc[ks][1], 8 * q4 + 4 + hs);
                const uint32_t b0 = even ? pack_h2(p0, p1) : 0u;
                const uint32_t b1 = even ? pack_h2(p2, p3) : 0u;
                const int tb = 16 * ks + 2 * q4;  // the lane's first token in the group
                const int nv = T - t0 - tb;       // tokens tb, tb + 1 valid if > 0, > 1; tb + 8, + 9 if > 8, > 9
                const uint32_t* vblk = st.v + ks * 64 * BITS;
#pragma unroll
                for (int j = 0; j < NGV; ++j) {  // V group j: m-tiles [8j / NGV, 8(j + 1) / NGV)
                    // (scale, zero) words of the lane's tokens; masked tokens may hold anything: zero them
                    const uint32_t w0 = nv > 0 ? st.vsz[tb * NGV + j] : 0u;
                    const uint32_t w1 = nv > 1 ? st.vsz[(tb + 1) * NGV + j] : 0u;
                    const uint32_t w2 = nv > 8 ? st.vsz[(tb + 8) * NGV + j] : 0u;
                    const uint32_t w3 = nv > 9 ? st.vsz[(tb + 9) * NGV + j] : 0u;
                    const uint32_t s01 = prmt(w0, w1, 0x5410u), z01 = prmt(w0, w1, 0x7632u);
                    const uint32_t s23 = prmt(w2, w3, 0x5410u), z23 = prmt(w2, w3, 0x7632u);
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        if (((mt * NGV) >> 3) != j) continue;  // resolved at compile time
                        uint32_t A[4];
                        v_pairs<BITS>(vblk + (8 * mt + g8) * BITS, q4, A);
                        mma16816(acc[mt], hfma2(A[0], s01, z01), hfma2(A[1], s01, z01), hfma2(A[2], s23, z23),
                                 hfma2(A[3], s23, z23), b0, b1);
                    }
                }
            }
        }
        __syncwarp();
        buf ^= 1;
    }
    cp_wait<0>();

    // ---- this warp's state per head: l summed over the head's eight lanes (g8)
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 4);
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 8);
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 16);
    if constexpr (VCOL) {
        // the zero-point sums of the columns: column n is summed over its four lanes 4n .. 4n + 3;
        // this lane's accumulator columns are 2 q4 and 2 q4 + 1
        zacc += __shfl_xor_sync(0xffffffffu, zacc, 1);
        zacc += __shfl_xor_sync(0xffffffffu, zacc, 2);
        const float z0 = __shfl_sync(0xffffffffu, zacc, 8 * q4);
        const float z1 = __shfl_sync(0xffffffffu, zacc, 8 * q4 + 4);
        __syncthreads();  // every warp is done with its stages: the union now holds the outputs
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int n = 2 * q4 + c, h = n / NGV;
            const int jc = NGV == 2 ? c : n % NGV;  // the column's V group
            const float z = c ? z1 : z0;
            if (h < GQ) {
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    if (((mt * NGV) >> 3) != jc) continue;
                    S.u.ro[warp][h][16 * mt + g8] = acc[mt][c] + z;
                    S.u.ro[warp][h][16 * mt + g8 + 8] = acc[mt][2 + c] + z;
                }
            }
        }
    } else {
        __syncthreads();  // every warp is done with its stages: the union now holds the outputs
        if (q4 < GQ) {
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                S.u.ro[warp][q4][16 * mt + g8] = acc[mt][0];
                S.u.ro[warp][q4][16 * mt + g8 + 8] = acc[mt][2];
            }
        }
    }
    if (g8 == 0 && q4 < GQ) {
        S.m[warp][q4] = mrun;
        S.l[warp][q4] = lrun;
    }
    __syncthreads();

    // ---- merge the warps, then the splits (the last CTA of the kv group)
    const int64_t rec0 = (((int64_t)b * Hv + gv) * a.n_splits + split) * GQ;
    for (int e = tid; e < GQ * D; e += NT) {
        const int h = e / D, d = e % D;
        float M = -INFINITY;
        for (int w = 0; w < NWARP; ++w) M = fmaxf(M, S.m[w][h]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
            for (int w = 0; w < NWARP; ++w) {
                const float wt = exp2f(S.m[w][h] - M);
                L = fmaf(S.l[w][h], wt, L);
                O = fmaf(S.u.ro[w][h][d], wt, O);
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
        const int prev = atomicAdd(&a.counters[b * Hv + gv], 1);
        is_last = (prev == nsplit_b - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    for (int e = tid; e < GQ * D; e += NT) {
        const int h = e / D, d = e % D;
        float M = -INFINITY;
        for (int sp = 0; sp < nsplit_b; ++sp)
            M = fmaxf(M, __ldcg(a.part + ((((int64_t)b * Hv + gv) * a.n_splits + sp) * GQ + h) * REC));
        float Lsum = 0.0f, acc2 = 0.0f;
        if (M != -INFINITY) {
            for (int sp = 0; sp < nsplit_b; ++sp) {
                const float* r = a.part + ((((int64_t)b * Hv + gv) * a.n_splits + sp) * GQ + h) * REC;
                const float w = exp2f(__ldcg(r) - M);
                Lsum = fmaf(__ldcg(r + 1), w, Lsum);
                acc2 = fmaf(__ldcg(r + 4 + d), w, acc2);
            }
        }
        a.out[((int64_t)b * Hq + gv * GQ + h) * D + d] = Lsum > 0.0f ? acc2 / Lsum : 0.0f;
    }
    if (tid == 0) a.counters[b * Hv + gv] = 0;
}

// ---------------------------------------------------------------- FP8 E4M3 layer
//
// K and V rows are E4M3 bytes (128 per token and kv head).  A warp takes 32 tokens (two pages) at
// a time; lane 0 stages the two pages of K and of V (four 2 KB blocks, contiguous per page and
// kv head) into the warp's shared-memory stage with bulk asynchronous copies that complete on the
// stage's mbarrier, one step ahead (two stages per warp).  E4M3 widens to fp16 exactly, so the
// scores are m16n8k16 products of exact fp16 keys with the fp16 query (exact products, fp32
// sums) and the values products of exact fp16 values with fp16 weights.  Channels are permuted
// inside each product (a dot product does not depend on the order), so that every lane reads
// whole 16-byte runs: in the score product lane q4 takes channels 32 q4 .. 32 q4 + 31 of a key
// row (k-step s: channels 32 q4 + 4 s + 0..3), in the value product output row (m-tile mt, g8)
// is channel 16 g8 + 2 mt and (mt, g8 + 8) channel 16 g8 + 2 mt + 1.  Head h of the kv group is
// column 2h of both products (odd columns zero), as in the code kernel above.

constexpr int F8_NW = 12;                 // warps per CTA (one CTA per SM)
constexpr int F8_NS = 2;                  // stages per warp (F8_NS - 1 steps in flight ahead of the one in use)
constexpr int F8_PAGE = PG * D;           // bytes of one page of one kv head (2 KB)
constexpr int F8_STAGE = 4 * F8_PAGE;     // K page 0, K page 1, V page 0, V page 1
constexpr uint32_t F8_SPIN = 1u << 16;    // bound on the polls of one mbarrier wait

template <int GQ>
struct F8Smem {
    union alignas(16) {
        uint8_t st[F8_NW][F8_NS][F8_STAGE];  // per warp: F8_NS stages
        float ro[F8_NW][GQ][D];           // per warp: unnormalised outputs, after the last step
    } u;
    unsigned long long bar[F8_NW][F8_NS];  // one mbarrier per stage (one arrival + the copied bytes)
    float m[F8_NW][GQ], l[F8_NW][GQ];
};

__device__ __forceinline__ uint32_t f8_saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void f8_expect(unsigned long long* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(f8_saddr(bar)), "r"(bytes)
                 : "memory");
}
// global -> shared bulk copy (16-byte aligned, a multiple of 16 bytes), completing on bar
__device__ __forceinline__ void f8_bulk(void* dst, const void* src, uint32_t bytes, unsigned long long* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     f8_saddr(dst)),
                 "l"(src), "r"(bytes), "r"(f8_saddr(bar))
                 : "memory");
}
// waits for the phase of bar with the given parity; false after F8_SPIN polls
__device__ __forceinline__ bool f8_wait(unsigned long long* bar, uint32_t parity) {
    for (uint32_t it = 0; it < F8_SPIN; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(f8_saddr(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}
// E4M3 x2 (low / high 16 bits of w) -> f16x2, exact
__device__ __forceinline__ uint32_t f8_lo(uint32_t w) {
    uint32_t r;
    asm("{\n.reg .b16 a, b;\nmov.b32 {a, b}, %1;\ncvt.rn.f16x2.e4m3x2 %0, a;\n}" : "=r"(r) : "r"(w));
    return r;
}
__device__ __forceinline__ uint32_t f8_hi(uint32_t w) {
    uint32_t r;
    asm("{\n.reg .b16 a, b;\nmov.b32 {a, b}, %1;\ncvt.rn.f16x2.e4m3x2 %0, b;\n}" : "=r"(r) : "r"(w));
    return r;
}
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }

template <int GQ>
__global__ void __launch_bounds__(32 * F8_NW, 1) f8_attn_kernel(QAttnArgs a) {
    constexpr int NT = 32 * F8_NW;
    static_assert(GQ <= 4, "at most four query heads per grid kv group");
    extern __shared__ __align__(16) unsigned char f8raw[];  // 16-byte aligned: every bulk copy's target is
    F8Smem<GQ>& S = *reinterpret_cast<F8Smem<GQ>*>(f8raw);   // at a multiple of 2 KB from it
    __shared__ int is_last;

    const int split = blockIdx.x, gv = blockIdx.y, b = blockIdx.z;
    const int Hv = gridDim.y, Hq = Hv * GQ;
    const int gk = gv / a.kv_div;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, q4 = lane & 3;
    if (tid < F8_NS * F8_NW) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(f8_saddr(&S.bar[tid / F8_NS][tid % F8_NS]))
                     : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    kvq_pdl_begin();
    const int T = a.seq_lens[b];
    if (T > a.max_len || T < 0) {
        if (tid == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_LENGTH, b);
        return;
    }
    const int n_groups = (T + KG - 1) / KG;
    const int n_pages = (T + PG - 1) / PG;
    const int nsplit_b = (n_groups + a.cps - 1) / a.cps;
    if (n_groups == 0) {
        if (split == 0)
            for (int i = tid; i < GQ * D; i += NT) a.out[((int64_t)b * Hq + gv * GQ) * D + i] = 0.0f;
        return;
    }
    if (split >= nsplit_b) return;
    const int hb = 2 * split * a.cps;                                   // this split's 32-token steps
    const int he = min(2 * min(n_groups, (split + 1) * a.cps), (n_pages + 1) / 2);

    // the query as the B operand of the score product: column 2h = head h (fp16, unscaled)
    const int hs = g8 >> 1;
    const bool qcol = (g8 & 1) == 0 && hs < GQ;
    uint32_t qb[8][2];
    {
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(a.q + ((int64_t)b * Hq + gv * GQ + (qcol ? hs : 0)) * D);
#pragma unroll
        for (int st = 0; st < 8; ++st) {
            qb[st][0] = qcol ? qw[16 * q4 + 2 * st] : 0u;
            qb[st][1] = qcol ? qw[16 * q4 + 2 * st + 1] : 0u;
        }
    }
    float acc[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][i] = 0.0f;
    float mrun = -INFINITY, lrun = 0.0f;
    bool ok_run = true;

    // lane 0: stage step j (tokens 32 j .. 32 j + 31) into stage stg of this warp
    auto issue = [&](int j, int stg) {
        uint8_t* dst = S.u.st[warp][stg];
        uint32_t bytes = 0;
        int32_t pg[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int lp = 2 * j + u;
            pg[u] = lp < n_pages ? a.bt[(int64_t)b * a.max_blocks + lp] : -1;
            if (lp < n_pages && (pg[u] < 0 || pg[u] >= a.num_blocks)) {
                kvq_dev_flag(a.hdr, KVQ_DEV_BAD_PAGE, b);
                pg[u] = -1;
            }
            if (pg[u] >= 0) bytes += 2 * F8_PAGE;
        }
        f8_expect(&S.bar[warp][stg], bytes);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (pg[u] < 0) continue;
            const int64_t off = ((int64_t)pg[u] * a.H + gk) * F8_PAGE;
            f8_bulk(dst + u * F8_PAGE, a.k_codes + off, F8_PAGE, &S.bar[warp][stg]);
            f8_bulk(dst + (2 + u) * F8_PAGE, a.v_codes + off, F8_PAGE, &S.bar[warp][stg]);
        }
    };

    int it = 0;
    if (lane == 0)
        for (int k = 0; k < F8_NS - 1; ++k)
            if (hb + warp + k * F8_NW < he) issue(hb + warp + k * F8_NW, k);
    for (int j = hb + warp; j < he; j += F8_NW, ++it) {
        const int stg = it % F8_NS;
        const int ahead = j + (F8_NS - 1) * F8_NW;
        if (lane == 0 && ahead < he) {
            // that stage was read in the previous step (ordered by the __syncwarp that ended it)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(ahead, (it + F8_NS - 1) % F8_NS);
        }
        if (!__all_sync(0xffffffffu, f8_wait(&S.bar[warp][stg], (uint32_t)(it / F8_NS) & 1u))) {  // warp-uniform
            if (lane == 0) kvq_dev_flag(a.hdr, KVQ_DEV_TIMEOUT, b);
            ok_run = false;
            break;
        }
        // pages of this step present in the stage (a page outside the pool was flagged, not copied)
        bool pv[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int lp = 2 * j + u;
            const int32_t pg = lp < n_pages ? a.bt[(int64_t)b * a.max_blocks + lp] : -1;
            pv[u] = pg >= 0 && pg < a.num_blocks;
        }
        const uint8_t* sb = S.u.st[warp][stg];
        const int t0 = 32 * j;

        // ---- scores: per page, rows g8 and g8 + 8 (head q4 in column 2 q4)
        float sc[2][2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const uint8_t* kp = sb + u * F8_PAGE + 32 * q4;
            const uint4 a0 = *reinterpret_cast<const uint4*>(kp + g8 * D);
            const uint4 a1 = *reinterpret_cast<const uint4*>(kp + g8 * D + 16);
            const uint4 b0 = *reinterpret_cast<const uint4*>(kp + (g8 + 8) * D);
            const uint4 b1 = *reinterpret_cast<const uint4*>(kp + (g8 + 8) * D + 16);
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int st = 0; st < 8; ++st) {
                const uint32_t wa = word_of(st < 4 ? a0 : a1, st & 3), wb = word_of(st < 4 ? b0 : b1, st & 3);
                mma16816(d, f8_lo(wa), f8_lo(wb), f8_hi(wa), f8_hi(wb), qb[st][0], qb[st][1]);
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = t0 + 16 * u + g8 + 8 * e;
                sc[u][e] = (pv[u] && t < T) ? d[2 * e] * KVQ_SCORE_LOG2_SCALE : -INFINITY;
            }
        }
        // ---- online softmax of head q4 over the step's 32 tokens
        float gm = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 4));
        gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 8));
        gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 16));
        const float mn = fmaxf(mrun, gm);
        const float alpha = mn == -INFINITY ? 1.0f : exp2f(mrun - mn);
        float ls = 0.0f;
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float p = mn == -INFINITY ? 0.0f : exp2f(sc[u][e] - mn);
                sc[u][e] = p;
                ls += p;
            }
        mrun = mn;
        lrun = fmaf(lrun, alpha, ls);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            acc[mt][0] *= alpha;
            acc[mt][2] *= alpha;
        }
        // ---- values, page by page: A = V^T (channels x tokens), B = p (column 2h = head h)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const float p0 = __shfl_sync(0xffffffffu, sc[u][0], 8 * q4 + hs);
            const float p1 = __shfl_sync(0xffffffffu, sc[u][0], 8 * q4 + 4 + hs);
            const float p2 = __shfl_sync(0xffffffffu, sc[u][1], 8 * q4 + hs);
            const float p3 = __shfl_sync(0xffffffffu, sc[u][1], 8 * q4 + 4 + hs);
            const uint32_t bb0 = qcol ? pack_h2(p0, p1) : 0u;
            const uint32_t bb1 = qcol ? pack_h2(p2, p3) : 0u;
            const uint8_t* vp = sb + (2 + u) * F8_PAGE + 16 * g8;
            const int tb = t0 + 16 * u + 2 * q4;  // the lane's first token
            // tokens past the sequence (or on a page that was not copied) hold anything: zero them
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            const uint4 vA = (pv[u] && tb < T) ? *reinterpret_cast<const uint4*>(vp + (2 * q4) * D) : z;
            const uint4 vB = (pv[u] && tb + 1 < T) ? *reinterpret_cast<const uint4*>(vp + (2 * q4 + 1) * D) : z;
            const uint4 vC = (pv[u] && tb + 8 < T) ? *reinterpret_cast<const uint4*>(vp + (2 * q4 + 8) * D) : z;
            const uint4 vE = (pv[u] && tb + 9 < T) ? *reinterpret_cast<const uint4*>(vp + (2 * q4 + 9) * D) : z;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;  // bytes 2k, 2k + 1 of two tokens, interleaved
                const uint32_t x01 = prmt(word_of(vA, mt >> 1), word_of(vB, mt >> 1), sel);
                const uint32_t x23 = prmt(word_of(vC, mt >> 1), word_of(vE, mt >> 1), sel);
                mma16816(acc[mt], f8_lo(x01), f8_hi(x01), f8_lo(x23), f8_hi(x23), bb0, bb1);
            }
        }
        __syncwarp();  // the stage is read: lane 0 may refill it
    }
    if (!ok_run && lane == 0) {
        // a wait that gave up: wait (bounded) for this warp's copies still in flight before the stage
        // memory goes away (the step it waited for, and the ones issued after it)
        for (int k = it; k < it + F8_NS; ++k)
            if (hb + warp + k * F8_NW < he) f8_wait(&S.bar[warp][k % F8_NS], (uint32_t)(k / F8_NS) & 1u);
    }

    // ---- this warp's state per head
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 4);
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 8);
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 16);
    __syncthreads();  // every warp is done with its stages: the union now holds the outputs
    if (q4 < GQ) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            S.u.ro[warp][q4][16 * g8 + 2 * mt] = acc[mt][0];
            S.u.ro[warp][q4][16 * g8 + 2 * mt + 1] = acc[mt][2];
        }
    }
    if (g8 == 0 && q4 < GQ) {
        S.m[warp][q4] = mrun;
        S.l[warp][q4] = lrun;
    }
    __syncthreads();

    // ---- merge the warps, then the splits (the last CTA of the kv group)
    const int64_t rec0 = (((int64_t)b * Hv + gv) * a.n_splits + split) * GQ;
    for (int e = tid; e < GQ * D; e += NT) {
        const int h = e / D, d = e % D;
        float M = -INFINITY;
        for (int w = 0; w < F8_NW; ++w) M = fmaxf(M, S.m[w][h]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
            for (int w = 0; w < F8_NW; ++w) {
                const float wt = exp2f(S.m[w][h] - M);
                L = fmaf(S.l[w][h], wt, L);
                O = fmaf(S.u.ro[w][h][d], wt, O);
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
        const int prev = atomicAdd(&a.counters[b * Hv + gv], 1);
        is_last = (prev == nsplit_b - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    for (int e = tid; e < GQ * D; e += NT) {
        const int h = e / D, d = e % D;
        float M = -INFINITY;
        for (int sp = 0; sp < nsplit_b; ++sp)
            M = fmaxf(M, __ldcg(a.part + ((((int64_t)b * Hv + gv) * a.n_splits + sp) * GQ + h) * REC));
        float Lsum = 0.0f, acc2 = 0.0f;
        if (M != -INFINITY) {
            for (int sp = 0; sp < nsplit_b; ++sp) {
                const float* r = a.part + ((((int64_t)b * Hv + gv) * a.n_splits + sp) * GQ + h) * REC;
                const float w = exp2f(__ldcg(r) - M);
                Lsum = fmaf(__ldcg(r + 1), w, Lsum);
                acc2 = fmaf(__ldcg(r + 4 + d), w, acc2);
            }
        }
        a.out[((int64_t)b * Hq + gv * GQ + h) * D + d] = Lsum > 0.0f ? acc2 / Lsum : 0.0f;
    }
    if (tid == 0) a.counters[b * Hv + gv] = 0;
}

// ---------------------------------------------------------------- planning and launch

// q heads per grid kv group: 8 sharing one kv head are served as two groups of 4
int grid_gq(int gq) { return gq > 4 ? 4 : gq; }
int kv_div_of(int gq) { return gq > 4 ? gq / 4 : 1; }

struct Plan {
    int n_splits;
    int cps;
};

template <int BITS, int GQ, int NGV>
int resident_one() {
    const int smem = (int)sizeof(QMSmem<BITS, GQ>);
    constexpr int NT = 32 * nwarp_of<BITS>();
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        kvq_prepare_kernel((const void*)qmma_kernel<BITS, GQ, NGV>, smem) == KVQ_OK &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, qmma_kernel<BITS, GQ, NGV>, NT, (size_t)smem) ==
            cudaSuccess &&
        n > 0)
        return n;
    cudaGetLastError();  // no device here: estimate from the thread and shared-memory budgets
    return std::max(1, std::min(2048 / NT, 232448 / (smem + 1024)));
}

template <int BITS, int GQ>
int resident_ngv(int G) {
    return G == 128 ? resident_one<BITS, GQ, 1>() : G == 64 ? resident_one<BITS, GQ, 2>() : resident_one<BITS, GQ, 4>();
}

template <int BITS>
int resident_bits(int gq, int G) {
    const int g = grid_gq(gq);
    return g == 1 ? resident_ngv<BITS, 1>(G) : g == 2 ? resident_ngv<BITS, 2>(G) : resident_ngv<BITS, 4>(G);
}

// CTAs of the layer's kernel that fit on one SM at once
int resident_ctas(const kvq_layout* L) {
    const int gq = L->n_q_heads / L->n_kv_heads, G = L->v_group_dims;
    if (kvq_code_bits(L) == KVQ_BITS_E4M3) return 1;  // the E4M3 kernel's stages fill an SM's shared memory
    switch (kvq_code_bits(L)) {
        case 1: return resident_bits<1>(gq, G);
        case 2: return resident_bits<2>(gq, G);
        case 4: return resident_bits<4>(gq, G);
        default: return resident_bits<8>(gq, G);
    }
}

// Context splits.  With few (sequence, kv head) units the split count fills one wave of resident
// CTAs.  With many units (a batch, lengths that may differ) every split takes a fixed 32 groups
// (2048 tokens), so a sequence gets CTAs in proportion to its length and the waves stay even;
// `compact` keeps the one-wave rule for callers with a small, fixed scratch.
constexpr int QA_SPLIT_GROUPS = 32;

Plan plan_splits(const kvq_layout* L, const kvq_seqs* S, bool compact) {
    const int n_groups = (std::max(S->max_len, 1) + KG - 1) / KG;
    const int gq = L->n_q_heads / L->n_kv_heads;
    const int64_t units = (int64_t)std::max(S->batch, 1) * L->n_kv_heads * kv_div_of(gq);
    const int64_t target = (int64_t)kvq_num_sms() * resident_ctas(L);  // one wave
    int cps;
    if (!compact && 2 * units >= target) {
        cps = std::min(n_groups, QA_SPLIT_GROUPS);
    } else {
        const int splits = (int)std::max<int64_t>(1, (target + units - 1) / units);
        cps = std::min(n_groups, std::max(4, (n_groups + splits - 1) / splits));
    }
    return {(n_groups + cps - 1) / cps, cps};
}

size_t ws_layout(const kvq_layout* L, const kvq_seqs* S, const Plan& p, size_t* off_part, size_t* off_cnt) {
    const int GQ = L->n_q_heads / L->n_kv_heads;
    const size_t units = (size_t)std::max(S->batch, 1) * L->n_kv_heads * kv_div_of(GQ);
    const size_t recs = units * p.n_splits * grid_gq(GQ);
    *off_part = sizeof(KvqWsHeader);
    *off_cnt = kvq_round_up(*off_part + recs * REC * sizeof(float), 256);
    return kvq_round_up(*off_cnt + units * sizeof(int32_t), 256);
}

template <int BITS, int GQ, int NGV, bool OUT = false>
int launch_one(dim3 grid, cudaStream_t s, const QAttnArgs& a) {
    const int smem = (int)(sizeof(QMSmem<BITS, GQ>) + (OUT ? ko_bytes<BITS>(a.n_out) : 0));
    static_assert(sizeof(QMSmem<BITS, 4>) + (OUT ? ko_bytes<BITS>(MAX_OUT) : 0) <= 227 * 1024,
                  "one CTA's stages fit in shared memory");
    const int st = kvq_prepare_kernel((const void*)qmma_kernel<BITS, GQ, NGV, OUT>, smem);
    if (st) return st;
    const cudaError_t e =
        kvq_launch_pdl(qmma_kernel<BITS, GQ, NGV, OUT>, grid, dim3(32 * nwarp_of<BITS>()), (size_t)smem, s, a);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_decode_attn_quant launch: %s", cudaGetErrorString(e));
    return KVQ_OK;
}

template <int BITS, int GQ, bool OUT = false>
int launch_ngv(dim3 grid, cudaStream_t s, const QAttnArgs& a) {
    switch (a.G) {
        case 128: return launch_one<BITS, GQ, 1, OUT>(grid, s, a);
        case 64: return launch_one<BITS, GQ, 2, OUT>(grid, s, a);
        default: return launch_one<BITS, GQ, 4, OUT>(grid, s, a);  // 32 (the only other size accepted)
    }
}

template <int GQ>
int launch_f8_gq(dim3 grid, cudaStream_t s, const QAttnArgs& a) {
    const int smem = (int)sizeof(F8Smem<GQ>);
    static_assert(sizeof(F8Smem<4>) <= 227 * 1024, "the E4M3 kernel's stages fit in shared memory");
    const int st = kvq_prepare_kernel((const void*)f8_attn_kernel<GQ>, smem);
    if (st) return st;
    const cudaError_t e = kvq_launch_pdl(f8_attn_kernel<GQ>, grid, dim3(32 * F8_NW), (size_t)smem, s, a);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_decode_attn_quant (E4M3) launch: %s", cudaGetErrorString(e));
    return KVQ_OK;
}

int launch_f8(int gq, dim3 grid, cudaStream_t s, QAttnArgs& a) {
    a.kv_div = kv_div_of(gq);
    grid.y *= a.kv_div;
    switch (grid_gq(gq)) {
        case 1: return launch_f8_gq<1>(grid, s, a);
        case 2: return launch_f8_gq<2>(grid, s, a);
        default: return launch_f8_gq<4>(grid, s, a);
    }
}

// grid: (splits, kv heads, batch); widened here to the grid kv groups
template <int BITS, bool OUT = false>
int launch_bits(int gq, dim3 grid, cudaStream_t s, QAttnArgs& a) {
    a.kv_div = kv_div_of(gq);
    grid.y *= a.kv_div;
    switch (grid_gq(gq)) {
        case 1: return launch_ngv<BITS, 1, OUT>(grid, s, a);
        case 2: return launch_ngv<BITS, 2, OUT>(grid, s, a);
        default: return launch_ngv<BITS, 4, OUT>(grid, s, a);
    }
}

// The bounded wait of the E4M3 kernel (f8_wait) on an mbarrier that nothing completes: one arrival
// is expected and none is made, so the phase never ends and the wait must give up.  Records
// KVQ_DEV_TIMEOUT, then returns: the diagnostic of kvq_selftest_bounded_wait.
__global__ void __launch_bounds__(32) f8_wait_selftest_kernel(KvqWsHeader* hdr) {
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x == 0) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(f8_saddr(&bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();
    if (!__all_sync(0xffffffffu, f8_wait(&bar, 0u)) && threadIdx.x == 0) kvq_dev_flag(hdr, KVQ_DEV_TIMEOUT, 0);
}

}  // namespace

extern "C" size_t kv_decode_attn_quant_ws(const kvq_layout* L, const kvq_seqs* S) {
    if (kvq_check_layout(L, "kv_decode_attn_quant_ws", true) || kvq_check_seqs_sizes(S, "kv_decode_attn_quant_ws"))
        return 0;
    size_t a, c;
    return ws_layout(L, S, plan_splits(L, S, false), &a, &c);
}

// The plan of the allocation-free variant: the default one if its scratch fits the built-in
// array, else the one-wave plan; NO_SPACE if neither fits.
static int noalloc_plan(const kvq_layout* L, const kvq_seqs* S, Plan* p, size_t* need, size_t* off_part,
                        size_t* off_cnt);

extern "C" int kv_decode_attn_quant_plan(const kvq_layout* L, const kvq_seqs* S, int32_t noalloc, int32_t* n_splits,
                                         int32_t* groups_per_split) {
    kvq_clear_error();
    int st = kvq_check_layout(L, "kv_decode_attn_quant_plan", true);
    if (st) return st;
    st = kvq_check_seqs_sizes(S, "kv_decode_attn_quant_plan");
    if (st) return st;
    KVQ_REQUIRE(n_splits && groups_per_split, KVQ_ERR_INVALID_ARG, "kv_decode_attn_quant_plan: NULL output");
    Plan p;
    if (noalloc) {
        size_t need, a, c;
        st = noalloc_plan(L, S, &p, &need, &a, &c);
        if (st) return st;
    } else {
        p = plan_splits(L, S, false);
    }
    *n_splits = p.n_splits;
    *groups_per_split = p.cps;
    return KVQ_OK;
}

// kv_decode_attn_quant and its outlier form; fn names the entry in messages.  k_out == NULL: the
// plain form.
static int decode_attn(const char* fn, const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q,
                       int32_t n_out, const int32_t* out_ch, const uint16_t* k_out, float* out, void* ws,
                       size_t ws_bytes, void* stream) {
    int st = kvq_check_layout(L, fn, true);
    if (st) return st;
    st = kvq_check_seqs(S, fn);
    if (st) return st;
    KVQ_REQUIRE(kvq_code_bits(L) != 16, KVQ_ERR_INVALID_ARG, "%s: layer is not quantized (bits == 16)", fn);
    KVQ_REQUIRE(P != nullptr && P->k_codes && P->v_codes &&
                    (kvq_code_bits(L) == KVQ_BITS_E4M3 || (P->k_sz && P->v_sz && P->k_tail)),
                KVQ_ERR_INVALID_ARG, "%s: quantized pool arrays missing", fn);
    KVQ_REQUIRE((((uintptr_t)P->k_codes | (uintptr_t)P->v_codes | (uintptr_t)P->k_sz | (uintptr_t)P->v_sz) & 15u) == 0,
                KVQ_ERR_INVALID_ARG, "%s: code and scale arrays must be 16-byte aligned", fn);
    KVQ_REQUIRE(S->batch <= P->max_seqs, KVQ_ERR_INVALID_ARG, "%s: batch exceeds max_seqs", fn);
    if (k_out) {
        const int cb = kvq_code_bits(L);
        KVQ_REQUIRE(cb == 4 || cb == 8, KVQ_ERR_UNSUPPORTED, "%s: isolated outlier channels need 4- or 8-bit codes",
                    fn);
        KVQ_REQUIRE(n_out >= 1 && n_out <= MAX_OUT && out_ch, KVQ_ERR_INVALID_ARG,
                    "%s: n_out %d not in [1, 8], or NULL out_ch", fn, n_out);
        KVQ_REQUIRE(((uintptr_t)k_out & 15u) == 0, KVQ_ERR_INVALID_ARG, "%s: k_out must be 16-byte aligned", fn);
    }
    size_t off_part, off_cnt;
    const Plan p = plan_splits(L, S, false);
    const size_t need = ws_layout(L, S, p, &off_part, &off_cnt);
    st = kvq_check_ws(ws, ws_bytes, need, fn);
    if (st) return st;
    if (S->batch == 0) return KVQ_OK;
    KVQ_REQUIRE(q && out && S->block_table, KVQ_ERR_INVALID_ARG, "%s: NULL q/out/block table", fn);
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
    a.k_out = k_out;
    a.out_ch = out_ch;
    a.n_out = k_out ? n_out : 0;
    const int gq = L->n_q_heads / L->n_kv_heads;
    dim3 grid(p.n_splits, L->n_kv_heads, S->batch);
    cudaStream_t s = kvq_stream(stream);
    if (k_out) {
        st = kvq_code_bits(L) == 4 ? launch_bits<4, true>(gq, grid, s, a) : launch_bits<8, true>(gq, grid, s, a);
    } else {
        switch (kvq_code_bits(L)) {
            case KVQ_BITS_E4M3: st = launch_f8(gq, grid, s, a); break;
            case 1: st = launch_bits<1>(gq, grid, s, a); break;
            case 2: st = launch_bits<2>(gq, grid, s, a); break;
            case 4: st = launch_bits<4>(gq, grid, s, a); break;
            default: st = launch_bits<8>(gq, grid, s, a); break;
        }
    }
    if (st) return st;
    return kvq_launch_status(fn);
}

extern "C" int kv_decode_attn_quant(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q,
                                    float* out, void* ws, size_t ws_bytes, void* stream) {
    kvq_clear_error();
    return decode_attn("kv_decode_attn_quant", L, P, S, q, 0, nullptr, nullptr, out, ws, ws_bytes, stream);
}

extern "C" int kv_decode_attn_quant_outlier(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S,
                                            const uint16_t* q, int32_t n_out, const int32_t* out_ch,
                                            const uint16_t* k_out, float* out, void* ws, size_t ws_bytes,
                                            void* stream) {
    kvq_clear_error();
    KVQ_REQUIRE(k_out, KVQ_ERR_INVALID_ARG, "kv_decode_attn_quant_outlier: NULL k_out");
    return decode_attn("kv_decode_attn_quant_outlier", L, P, S, q, n_out, out_ch, k_out, out, ws, ws_bytes, stream);
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

// Device address of g_qattn_scratch in the current context, looked up on every call (a host-side
// lookup; a cached address would go stale if the context were reset and the module reloaded).
static int qattn_scratch(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_qattn_scratch);
    if (e != cudaSuccess || p == nullptr)
        return kvq_fail(KVQ_ERR_CUDA, "kv_decode_attn_quant_noalloc: scratch address: %s", cudaGetErrorString(e));
    *out = p;
    return KVQ_OK;
}

extern "C" size_t kv_decode_attn_quant_noalloc_max_scratch(void) { return KVQ_NOALLOC_SCRATCH_BYTES; }

extern "C" int kvq_selftest_bounded_wait(void* ws, size_t ws_bytes, void* stream) {
    kvq_clear_error();
    int st = kvq_check_ws(ws, ws_bytes, sizeof(KvqWsHeader), "kvq_selftest_bounded_wait");
    if (st) return st;
    f8_wait_selftest_kernel<<<1, 32, 0, kvq_stream(stream)>>>(static_cast<KvqWsHeader*>(ws));
    return kvq_launch_status("kvq_selftest_bounded_wait");
}

static int noalloc_plan(const kvq_layout* L, const kvq_seqs* S, Plan* p, size_t* need, size_t* off_part,
                        size_t* off_cnt) {
    *p = plan_splits(L, S, false);
    *need = ws_layout(L, S, *p, off_part, off_cnt);
    if (*need > KVQ_NOALLOC_SCRATCH_BYTES) {  // fewer splits, if that fits
        *p = plan_splits(L, S, true);
        *need = ws_layout(L, S, *p, off_part, off_cnt);
    }
    KVQ_REQUIRE(*need <= KVQ_NOALLOC_SCRATCH_BYTES, KVQ_ERR_NO_SPACE,
                "kv_decode_attn_quant_noalloc: this batch needs %zu bytes of scratch, the built-in array holds %u; "
                "use kv_decode_attn_quant with a workspace", *need, KVQ_NOALLOC_SCRATCH_BYTES);
    return KVQ_OK;
}

extern "C" int kv_decode_attn_quant_noalloc(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S,
                                            const uint16_t* q, float* out, void* stream) {
    kvq_clear_error();
    int st = kvq_check_layout(L, "kv_decode_attn_quant_noalloc", true);
    if (st) return st;
    st = kvq_check_seqs(S, "kv_decode_attn_quant_noalloc");
    if (st) return st;
    KVQ_REQUIRE(kvq_code_bits(L) != 16, KVQ_ERR_INVALID_ARG, "kv_decode_attn_quant_noalloc: layer is not quantized");
    KVQ_REQUIRE(P != nullptr && P->k_codes && P->v_codes &&
                    (kvq_code_bits(L) == KVQ_BITS_E4M3 || (P->k_sz && P->v_sz && P->k_tail)),
                KVQ_ERR_INVALID_ARG, "kv_decode_attn_quant_noalloc: quantized pool arrays missing");
    KVQ_REQUIRE((((uintptr_t)P->k_codes | (uintptr_t)P->v_codes | (uintptr_t)P->k_sz | (uintptr_t)P->v_sz) & 15u) == 0,
                KVQ_ERR_INVALID_ARG, "kv_decode_attn_quant_noalloc: code and scale arrays must be 16-byte aligned");
    KVQ_REQUIRE(S->batch <= P->max_seqs, KVQ_ERR_INVALID_ARG, "kv_decode_attn_quant_noalloc: batch exceeds max_seqs");
    size_t off_part, off_cnt, need;
    Plan p;
    st = noalloc_plan(L, S, &p, &need, &off_part, &off_cnt);
    if (st) return st;
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
    switch (kvq_code_bits(L)) {
        case KVQ_BITS_E4M3: st = launch_f8(gq, grid, s, a); break;
        case 1: st = launch_bits<1>(gq, grid, s, a); break;
        case 2: st = launch_bits<2>(gq, grid, s, a); break;
        case 4: st = launch_bits<4>(gq, grid, s, a); break;
        default: st = launch_bits<8>(gq, grid, s, a); break;
    }
    if (st) return st;
    return kvq_launch_status("kv_decode_attn_quant_noalloc");
}
