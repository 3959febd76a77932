/*
 * kvq.h -- C ABI of libkvq: compressed-KV decode attention on one GB300 GPU.
 *
 * The library implements the decode-step hot path of a compressed KV cache:
 * asymmetric b-bit packing, paged 16-token blocks, fused dequant attention,
 * the sparse-layer path (critical-channel scores, top-K with sinks and a
 * recent window, exact attention over the selection), the H2O cumulative
 * score update and the dense-preference layer score; and around it the
 * host-link gather of offloaded rows, block-granular and GQA-shared
 * selection, a layer whose kv heads are classified one by one (dense or
 * sparse), isolated fp16 outlier key channels beside a quantized cache, an
 * FP8 E4M3 cache and symmetric V quantization.
 *
 * Sources cited below (page, then section):
 *   [TailorKV]  "TailorKV" article, ijyty.com/news/1204784
 *   [KVSurvey]  "大语言模型长上下文推理与KV Cache前沿压缩策略解析",
 *               bbs.huaweicloud.com/blogs/490932
 *   [OnDevice]  "端侧大模型KV缓存量化卸载协同：详解分层稀疏注意力与异构内存池动态迁移机制",
 *               ufo.work/2026/495
 *   [Meeting]   "长上下文会议大模型推理KV缓存稀疏化与量化联合压缩：剖析重要性评分指标与异构内存分层调度策略",
 *               ufo.work/2026/545
 *
 * Conventions shared by every call
 *   - Every function returns an int status: KVQ_OK (0) or a negative KVQ_ERR_*.
 *     kvq_last_error() returns a message for the calling thread's last failure.
 *   - Arguments are validated on the host before anything is launched; a
 *     rejected call launches nothing.
 *   - The caller owns every buffer.  The library never allocates or frees
 *     device memory.  Pointers documented "device" must be device-accessible
 *     (cudaMalloc / torch CUDA tensors); "host" pointers are ordinary memory;
 *     "mapped" pointers are pinned host memory the GPU can read.
 *   - Device calls are asynchronous on the given stream (a cudaStream_t passed
 *     as void*; NULL is the legacy default stream).
 *   - fp16 data is IEEE binary16 passed as uint16_t.  head_dim d is 128.
 *   - Workspaces ("ws") are device buffers of at least the size the matching
 *     *_ws() function returns, 256-byte aligned, ZERO-FILLED BEFORE FIRST USE.
 *     The library leaves them zeroed after every call that completes, so they
 *     can be reused; after a call that failed on the device, zero them again.
 *     The one exception is a handful of diagnostic path counters in the first
 *     256 bytes (kvq_read_path_counters), which kernels only add to and never
 *     read.  Two calls that share a workspace must not run concurrently.
 *   - Data-dependent device errors (a page id outside the pool, a selected id
 *     outside the sequence) skip the faulty access and set a status word in
 *     the workspace; kvq_check() reads and clears it.  Nothing traps, and no
 *     kernel waits on another CTA's flag: the only waits are bounded waits for
 *     a kernel's own asynchronous copies, which on expiry set the status word
 *     (KVQ_ERR_DEVICE_CHECK from kvq_check, "a bounded wait ... gave up").
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_OK                 0
#define KVQ_ERR_INVALID_ARG   -1
#define KVQ_ERR_UNSUPPORTED   -2
#define KVQ_ERR_CUDA          -3
#define KVQ_ERR_NO_SPACE      -4
#define KVQ_ERR_TIMEOUT       -5
#define KVQ_ERR_DEVICE_CHECK  -6

/* Diagnostic path counters in a workspace header (kvq_read_path_counters). */
#define KVQ_N_PATH_COUNTERS    4
#define KVQ_PATH_LISTED        0  /* sparse-layer CTAs that attended their kept rows from the
                                     one-pass list (no ordered compaction) */
#define KVQ_PATH_COMPACTED     1  /* sparse-layer CTAs that compacted their kept positions in order
                                     (a `sel` output, everything kept, or a list overflow) */
#define KVQ_PATH_RADIX_PASSES  2  /* selections (clusters) whose first-digit candidates overflowed
                                     their slots and took distributed radix passes */
#define KVQ_PATH_RESERVED      3

/* kvq_layout.bits of an FP8 E4M3 layer: K and V rows cast to E4M3 bytes (round
 * to nearest even, finite values saturate at +-448), 128 bytes per token and kv
 * head, no scales [Meeting §6 item 2: FP8 E4M3 preferred where the hardware
 * has it, no dequantization arithmetic]. */
#define KVQ_BITS_E4M3         0xE4

/* Or-ed into kvq_layout.bits of a 2-, 4- or 8-bit layer: V is quantized
 * symmetrically [OnDevice §3.1: V INT4 symmetric, group quantization]: per token
 * and V group, scale = max|x| / L with L = 2^(b-1) - 1, code = clamp(round(x /
 * scale), -L, L) (fp32, round half to even), scale stored fp16.  The page layout
 * is the asymmetric one with the code stored as code + L and the (scale, zero)
 * pair as (scale16, fp16(-L * scale16)), so attention reads it unchanged. */
#define KVQ_V_SYMMETRIC       0x100

#define KVQ_HEAD_DIM          128
#define KVQ_BLOCK_TOKENS      16
#define KVQ_K_GROUP_TOKENS    64

/* Thread-local text of the last error of the calling thread ("" if none). */
const char* kvq_last_error(void);

/* ABI version; bumped whenever a struct or signature below changes. */
int kvq_version(void);

/* ------------------------------------------------------------------------
 * Descriptors (plain structs, passed by host pointer, read during the call).
 * ---------------------------------------------------------------------- */

/* Geometry of one layer's cache. */
typedef struct kvq_layout {
    int32_t head_dim;        /* d; must be 128 */
    int32_t n_q_heads;       /* H_q; a multiple of n_kv_heads, H_q / H_kv <= 8 */
    int32_t n_kv_heads;      /* H_kv; q head h reads kv head floor(h * H_kv / H_q) */
    int32_t block_tokens;    /* tokens per page; must be 16 [KVSurvey §一.1] */
    int32_t bits;            /* 1, 2, 4, 8: quantized layer (2, 4, 8 may carry
                                KVQ_V_SYMMETRIC); 16: fp16 layer;
                                KVQ_BITS_E4M3: FP8 E4M3 layer */
    int32_t k_group_tokens;  /* K quantization group along tokens; must be 64 [TailorKV §2.2] */
    int32_t v_group_dims;    /* V quantization group along head_dim: 32, 64 or 128 [OnDevice §3.1] */
} kvq_layout;

/* Device storage of one layer.  Fields a layer kind does not use may be NULL.
 * Pages are indexed by physical page id p in [0, num_blocks); per-sequence
 * state is indexed by the sequence's batch index b in [0, max_seqs).
 *
 * Quantized layer (bits in {1,2,4,8}); R = d*bits/8 bytes per token row;
 * blocks are read as little-endian 32-bit words, n = 16/bits codes per half
 * word, and codes travel in pairs: the two codes of a pair sit at the same
 * offset o in the low and the high half of one word (bits [o, o+bits) and
 * [16+o, 16+o+bits)), the layout the tensor-core fragments read:
 *   k_codes [num_blocks][H_kv][16][R]   uint8; K codes, one row per token.
 *     Channels (2p, 2p+1), p = 8s + r + 4e (s < 8, r < 4, e < 2), form pair
 *     m = 2s + e of column r: word r*bits + m/n of the row, o = (m%n)*bits,
 *     the odd channel in the high half.
 *   v_codes [num_blocks][H_kv][16][R]   uint8; V codes, one 16*R-byte block
 *     per page and kv head, channel-major: channel d = 16t + 8u + x
 *     (x < 8, u < 2) and the page's tokens (2y, 2y+1), y = r + 4e (r < 4,
 *     e < 2), form pair m = 4r + 2e + u of row 8t + x: word
 *     (8t + x)*bits + m/n of the block, o = (m%n)*bits, the odd token in the
 *     high half.
 *   k_sz    [num_blocks][H_kv][d][2]    fp16 (scale, zero) of the 64-token K
 *           group whose FIRST page is p (entries of other pages are unused)
 *   v_sz    [num_blocks][H_kv][16][d/G][2]  fp16 (scale, zero) per token and
 *           V group of G = v_group_dims channels
 *   k_tail  [max_seqs][H_kv][64][d]     fp16 keys of the unfinished K group
 *           (tokens 64*floor(T/64) .. T-1 at rows t mod 64)
 * FP8 E4M3 layer (bits == KVQ_BITS_E4M3):
 *   k_codes, v_codes [num_blocks][H_kv][16][d] E4M3 bytes of the K and V rows
 *   (k_sz, v_sz, k_tail unused)
 * fp16 layer (bits == 16):
 *   k16, v16 [num_blocks][H_kv][16][d]  fp16 token rows
 *   kT       [max_seqs][H_kv][d][t_cap] fp16 channel-major copy of K, the
 *            "critical key" buffer read by kv_critical_score (t_cap % 8 == 0;
 *            kv_sparse_layer_decode also needs t_cap <= 2^24)
 *   k_absmax [max_seqs][H_kv][d]        fp32 running max_t |K[t][c]|
 *            (kT and k_absmax may both be NULL for a layer that is never
 *            scored, e.g. an H2O layer; pack and append then skip them)
 */
typedef struct kvq_pool {
    int64_t   num_blocks;
    int32_t   max_seqs;
    int32_t   t_cap;
    uint8_t*  k_codes;
    uint8_t*  v_codes;
    uint16_t* k_sz;
    uint16_t* v_sz;
    uint16_t* k_tail;
    uint16_t* k16;
    uint16_t* v16;
    uint16_t* kT;
    float*    k_absmax;
} kvq_pool;

/* The batch of sequences a call works on.  Sequence b owns pool slot b. */
typedef struct kvq_seqs {
    const int32_t* block_table;  /* device [batch][max_blocks]: physical page of
                                    logical page j (tokens 16j..16j+15) */
    const int32_t* seq_lens;     /* device [batch]: tokens in the cache, counting
                                    the newest one */
    int32_t batch;               /* B <= max_seqs */
    int32_t max_blocks;          /* row stride of block_table */
    int32_t max_len;             /* host upper bound on every seq_lens[b]; sizes
                                    grids and workspaces (<= 16 * max_blocks) */
    int32_t reserved;
} kvq_seqs;

/* ------------------------------------------------------------------------
 * a1: kv_quant_pack -- write a run of prompt tokens into a layer's cache.
 * [TailorKV §2.2] scale = (max - min)/(2^b - 1), zero = min,
 * code = clamp(round((x - zero)/scale), 0, 2^b - 1), scale/zero kept as fp16;
 * K per channel over 64-token groups, V per token over G-channel groups
 * [OnDevice §3.1].  Arithmetic: IEEE fp32 on fp16 inputs, codes computed
 * with the fp32 scale, round half to even; a group with max == min gets
 * scale 0 and codes 0.
 *
 * An FP8 E4M3 layer (bits == KVQ_BITS_E4M3) stores every K and V value as an
 * E4M3 byte (cvt with round-to-nearest-even, saturating), no scales.
 *
 * Writes tokens t_start .. t_start+n_tokens-1 of sequence `seq`.  k and v are
 * device fp16 [n_tokens][H_kv][d] with `stride_t` elements between tokens
 * (>= H_kv*d).  t_start must be a multiple of 64.  Complete 64-token K groups
 * are quantized into k_codes/k_sz; the keys of a final partial group go to
 * k_tail; every token's V is quantized.  For an fp16 layer (bits == 16) the
 * rows go to k16/v16, kT and k_absmax (absmax is raised, never lowered).
 * Pages block_table[seq][t/16] must be allocated.  No workspace.
 * Errors: INVALID_ARG (NULL/shape/alignment), UNSUPPORTED (d, bits, G), CUDA.
 * ---------------------------------------------------------------------- */
int kv_quant_pack(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                  int32_t seq, int64_t t_start, int64_t n_tokens,
                  const uint16_t* k, const uint16_t* v, int64_t stride_t,
                  void* stream);

/* ------------------------------------------------------------------------
 * a2: kv_page_append -- append one decode token to every sequence.
 * [KVSurvey §一.1] paged blocks of 16 tokens through a per-sequence block
 * table; quantization as in kv_quant_pack.
 *
 * k_new, v_new: device fp16 [batch][H_kv][d].  The token is written at
 * position seq_lens[b] - 1 (seq_lens already counts it; see kvq_seq_lens_add).
 * Quantized layer: V is quantized at once; K goes to k_tail and, when it
 * completes a 64-token group, the group is quantized into its four pages.
 * fp16 layer: the rows go to k16/v16, kT and k_absmax.
 * The page of the new token must be allocated and not shared (copy it first
 * with kv_page_copy if its reference count is above one).
 * ws: kv_page_append_ws() bytes (status word only).
 * ---------------------------------------------------------------------- */
int kv_page_append(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                   const uint16_t* k_new, const uint16_t* v_new,
                   void* ws, size_t ws_bytes, void* stream);
size_t kv_page_append_ws(void);

/* ------------------------------------------------------------------------
 * a3: kv_decode_attn_quant -- fused dequant -> q.k/sqrt(d) -> softmax -> p.v
 * over the quantized cache [OnDevice §3.2; TailorKV §2.2].
 *
 * q: device fp16 [batch][H_q][d]; out: device fp32 [batch][H_q][d].
 * Packed tokens use dequantized K (zero + code*scale with the stored fp16
 * scale/zero); tail tokens use their fp16 keys exactly; V is dequantized.
 * Both products run on the tensor cores with fp32 accumulation: q*scale
 * enters as two fp16 halves (about 22 bits); for the values, either (heads
 * per kv head times V groups per token <= 8) the V codes enter exactly against
 * fp16(2^8 p * vscale) per token, with the zero points summed in fp32, or (4
 * heads with 32-dim V groups) the dequantized V rows against the softmax
 * weights, both fp16 (relative rounding 2^-11 per element, averaging out over
 * the tokens).  |q_c * scale_c| * 2^bits must stay below 32768 and, on the
 * first form, |vscale| below 256 (the fp16 operand range); otherwise the
 * status word reports a range error and the output is not valid.  The context is split across CTAs and the
 * partial softmax states are merged by log-sum-exp.  An empty sequence gives 0.
 * An FP8 E4M3 layer (bits == KVQ_BITS_E4M3) is attended the same way: its
 * pages are staged into shared memory by bulk asynchronous copies, keys and
 * values widened to fp16 (exactly) for the tensor cores; products with q are
 * exact, sums fp32, p enters the value product in fp16.
 * ws: kv_decode_attn_quant_ws(layout, seqs) bytes.
 * ---------------------------------------------------------------------- */
int kv_decode_attn_quant(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                         const uint16_t* q, float* out,
                         void* ws, size_t ws_bytes, void* stream);
size_t kv_decode_attn_quant_ws(const kvq_layout* layout, const kvq_seqs* seqs);

/* ------------------------------------------------------------------------
 * kv_decode_attn_quant_noalloc -- kv_decode_attn_quant without a workspace.
 * (An addition of this library: the pages describe no such call.)
 *
 * For callers that cannot hand the library device memory: a plugin whose host
 * framework owns every allocation and passes only input and output buffers,
 * or a decode loop that must never enter the CUDA allocator (cudaMalloc can
 * synchronize the device).  It computes exactly what kv_decode_attn_quant
 * computes, with the same arguments minus the workspace; the split-K scratch
 * is one fixed 8 MiB array inside the library (kv_decode_attn_quant_noalloc_
 * max_scratch() bytes), which every GPU that loads the library keeps until
 * the process exits.  No call allocates or frees memory.
 *   - Every call looks up the array's device address in the current context
 *     (a host-side lookup, so a context reset leaves no stale address); the
 *     first call on a device loads the array's module, so make it before any
 *     stream capture.
 *   - A batch whose scratch (kv_decode_attn_quant_ws) exceeds the array is
 *     rejected with KVQ_ERR_NO_SPACE before anything is launched.
 *   - All calls share the array and each clears the parts that must start at
 *     zero; calls that overlap on the GPU (other streams, other threads) race
 *     and give wrong results.  Device data checks still skip bad accesses, but
 *     their status word is not reported (there is no workspace for kvq_check).
 * ---------------------------------------------------------------------- */
int kv_decode_attn_quant_noalloc(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                                 const uint16_t* q, float* out, void* stream);
size_t kv_decode_attn_quant_noalloc_max_scratch(void);

/* The split of the context kv_decode_attn_quant (noalloc == 0) or
 * kv_decode_attn_quant_noalloc (noalloc != 0) uses for this layout and batch:
 * *n_splits CTAs per (sequence, group of up to 4 q heads), each taking
 * *groups_per_split consecutive 64-token groups.  Host only; no launch.
 * Errors: INVALID_ARG / UNSUPPORTED as the attention call would report;
 * NO_SPACE for a noalloc batch beyond the built-in array. */
int kv_decode_attn_quant_plan(const kvq_layout* layout, const kvq_seqs* seqs, int32_t noalloc,
                              int32_t* n_splits, int32_t* groups_per_split);

/* ------------------------------------------------------------------------
 * f3: outlier-channel isolation of the keys [Meeting §8.2: the channels of
 * largest variance per layer and head kept in fp16 beside a quantized main
 * cache, and a single fused attention kernel over both].
 *
 * Outlier channels are chosen per (sequence, kv head) from that sequence's
 * prompt keys; the main cache is the layer's ordinary cache (kv_quant_pack /
 * kv_page_append) in which those channels' codes, K scale and K zero are then
 * set to 0, and their fp16 keys are kept in a side cache
 *   k_out   [num_blocks][H_kv][16][n_out]  fp16, rows of packed tokens only
 *           (tail tokens keep every channel in k_tail)
 *   out_ch  [batch][H_kv][n_out]           int32, ascending channels of the
 *           sequence in batch slot b
 * 1 <= n_out <= 8; only 4- and 8-bit layers (the page's INT4 main cache, and
 * 8 bits).  k_out rows and page rows follow the same block table.  V is not
 * split.  An isolated cache must be attended with kv_decode_attn_quant_outlier
 * (kv_decode_attn_quant would omit the outlier channels).
 * ---------------------------------------------------------------------- */

/* kv_outlier_channels: the n_out channels of largest variance per kv head of
 * n_tokens fp16 keys k [n_tokens][H_kv][d] (device, `stride_t` elements
 * between tokens, finite values).  Var_c = (S2 - S1^2/T)/T in fp64 from the
 * exact sums S1 = sum K[t][c], S2 = sum K[t][c]^2 (integer arithmetic: fp16
 * values are multiples of 2^-24), each rounded once to fp64; one rounding per
 * operation after that.  Ties -> lower channel.  out_ch: device int32
 * [H_kv][n_out], ascending.  var (optional, may be NULL): device fp64
 * [H_kv][d].  n_tokens <= 2^22; n_tokens == 0 gives variance 0 and channels
 * 0 .. n_out-1.  ws: kv_outlier_channels_ws(layout) bytes, zeroed before the
 * first call; the call leaves it zeroed.  Errors: INVALID_ARG, CUDA. */
int kv_outlier_channels(const kvq_layout* layout, const uint16_t* k, int64_t n_tokens, int64_t stride_t,
                        int32_t n_out, int32_t* out_ch, double* var, void* ws, size_t ws_bytes,
                        void* stream);
size_t kv_outlier_channels_ws(const kvq_layout* layout);

/* kv_outlier_isolate: after kv_quant_pack of tokens t_start .. t_start +
 * n_tokens - 1 of sequence `seq` (the same k, stride_t), isolates the outlier
 * channels out_ch[seq] of every complete 64-token group of that run: their
 * fp16 keys into k_out, their codes in k_codes and their (scale, zero) in
 * k_sz set to 0.  A final partial group stays in k_tail (all channels fp16)
 * and is isolated by kv_outlier_append when it completes.  t_start must be a
 * multiple of 64.  No workspace; device checks skip bad pages or channels
 * without a status word.  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
int kv_outlier_isolate(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                       int32_t seq, int64_t t_start, int64_t n_tokens, const uint16_t* k, int64_t stride_t,
                       int32_t n_out, const int32_t* out_ch, uint16_t* k_out, void* stream);

/* kv_outlier_append: after kv_page_append, for every sequence whose new token
 * completed a 64-token K group (seq_lens[b] % 64 == 0), isolates the outlier
 * channels of that group (keys read from k_tail).  Run it after every append
 * of an isolated layer, before the next append.  ws: kv_outlier_append_ws()
 * bytes (status word: bad page or channel). */
int kv_outlier_append(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                      int32_t n_out, const int32_t* out_ch, uint16_t* k_out,
                      void* ws, size_t ws_bytes, void* stream);
size_t kv_outlier_append_ws(void);

/* kv_decode_attn_quant_outlier: kv_decode_attn_quant over an isolated cache.
 * Packed tokens' scores add sum_j q[c_j] * k_out[t][j] (fp16 products, exact
 * in fp32, summed in fp32) to the main cache's score, inside the same kernel:
 * the outlier keys of a 64-token group are staged into shared memory beside
 * its codes.  k_out 16-byte aligned.  ws: kv_decode_attn_quant_ws(layout,
 * seqs) bytes.  Errors as kv_decode_attn_quant; UNSUPPORTED for bits other
 * than 4 and 8. */
int kv_decode_attn_quant_outlier(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                                 const uint16_t* q, int32_t n_out, const int32_t* out_ch,
                                 const uint16_t* k_out, float* out,
                                 void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * a4: kv_critical_score -- approximate token scores from critical channels
 * [TailorKV §2.3]: s_c = |q_c| * max_t |K[t][c]| picks the n_crit channels
 * with the largest s_c (ties -> lower channel); then for every cached token
 * a_t = sum over those channels, in ascending channel order, of q_c*K[t][c],
 * in fp32 starting from +0.
 *
 * Reads kT and k_absmax of an fp16 layer.  q: device fp16 [batch][H_q][d].
 * crit (optional, may be NULL): device int32 [batch][H_q][n_crit], ascending.
 * scores: device fp32 [batch][H_q][score_stride], entries t < seq_lens[b]
 * written.  1 <= n_crit <= 128; score_stride >= max_len, multiple of 4.
 * ---------------------------------------------------------------------- */
int kv_critical_score(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                      const uint16_t* q, int32_t n_crit, int32_t* crit,
                      float* scores, int64_t score_stride, void* stream);

/* ------------------------------------------------------------------------
 * f1: kv_group_critical_score -- kv_critical_score shared by the query heads
 * of one kv head (GQA) [TailorKV §2.3 applied per kv head; Meeting §8.1 item 1].
 * Reading (the pages say only "the query"): a channel's importance for kv head
 * g is (sum over g's q heads, ascending, of |q_h,c|, fp32) * max_t |K[t][c]|
 * (fp32); the n_crit largest (ties -> lower channel) are the group's channels;
 * a token's score is the fp32 sum, in ascending head order, of each head's
 * approximate score on those channels (as kv_critical_score computes it).
 * One selection per kv head then serves all its q heads: kv_topk_select with
 * n_heads = H_kv, kv_sparse_attn with sel_per_kv_head = 1 -- the channel rows,
 * the selection and the selected rows are read once per kv head instead of
 * once per q head.
 *
 * q: device fp16 [batch][H_q][d]; crit (optional): device int32
 * [batch][H_kv][n_crit], ascending; scores: device fp32
 * [batch][H_kv][score_stride].  Otherwise as kv_critical_score.
 * ---------------------------------------------------------------------- */
int kv_group_critical_score(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                            const uint16_t* q, int32_t n_crit, int32_t* crit,
                            float* scores, int64_t score_stride, void* stream);

/* ------------------------------------------------------------------------
 * a5: kv_topk_select -- token selection per query head [TailorKV §2.3, §5.1;
 * KVSurvey §三.1]: tokens [0, n_sink) and [T-window, T) are always kept;
 * among the others the k highest scores (ties -> lower position) are added;
 * if n_sink + window + k >= T every token is kept.  Output ids ascending.
 *
 * scores: device fp32 [batch][n_heads][score_stride].  k = k_fixed when
 * k_fixed >= 0, else floor(ratio * T) computed in double with T = seq_lens[b].
 * sel: device int32 [batch][n_heads][sel_cap]; sel_count: device int32
 * [batch][n_heads].  sel_cap must hold the largest selection.
 * T <= 8 * 45056 = 360448 per call (UNSUPPORTED above).
 * ws: kv_topk_select_ws() bytes (status word only).
 * ---------------------------------------------------------------------- */
int kv_topk_select(const kvq_seqs* seqs, int32_t n_heads,
                   const float* scores, int64_t score_stride,
                   int32_t k_fixed, double ratio, int32_t n_sink, int32_t window,
                   int32_t* sel, int32_t sel_cap, int32_t* sel_count,
                   void* ws, size_t ws_bytes, void* stream);
size_t kv_topk_select_ws(void);

/* ------------------------------------------------------------------------
 * f1: kv_block_select -- block-granular selection, the block pruning of
 * the meeting article [Meeting §8.1, item 1]: tokens are grouped into
 * blocks of block_tokens (block j = tokens [j*block, (j+1)*block) of the
 * sequence); a block's importance is the mean score of its candidate
 * tokens (n_sink <= t < T - window): an fp32 sum in ascending t divided
 * by the count in fp32 (-inf without candidates).  The n blocks of highest importance (ties -> lower block)
 * are kept whole, with n = n_keep_fixed when >= 0, else
 * floor(ratio * ceil(T / block)) in double.  Output: the sinks [0, n_sink),
 * every token of the kept blocks and the window [T - window, T), as
 * ascending ids; feeds kv_sparse_attn (contiguous runs of rows).
 *
 * scores: device fp32 [batch][n_heads][score_stride] (score_stride >=
 * max_len).  sel: device int32 [batch][n_heads][sel_cap]; sel_count: device
 * int32 [batch][n_heads]; a selection larger than sel_cap is cut and flags
 * KVQ_DEV_OVERFLOW.  ceil(max_len / block) <= 24576 (UNSUPPORTED above).
 * Two launches (the importances; the choice of blocks and the token ids).
 * ws: kv_block_select_ws(seqs, n_heads, block_tokens) bytes.
 * ---------------------------------------------------------------------- */
int kv_block_select(const kvq_seqs* seqs, int32_t n_heads,
                    const float* scores, int64_t score_stride,
                    int32_t n_keep_fixed, double ratio, int32_t n_sink, int32_t window,
                    int32_t block_tokens, int32_t* sel, int32_t sel_cap, int32_t* sel_count,
                    void* ws, size_t ws_bytes, void* stream);
size_t kv_block_select_ws(const kvq_seqs* seqs, int32_t n_heads, int32_t block_tokens);

/* ------------------------------------------------------------------------
 * a6: kv_sparse_attn -- exact softmax attention over selected tokens
 * [Meeting §3.2: Softmax(Q K_ret^T / sqrt(d)) V_ret; Meeting §8.1].
 *
 * Reads fp16 rows k16/v16 through the block table.  q: device fp16
 * [batch][H_q][d]; out: device fp32 [batch][H_q][d].
 * sel_per_kv_head == 0: sel is [batch][H_q][sel_cap], one list per q head;
 * sel_per_kv_head == 1: sel is [batch][H_kv][sel_cap], shared by the q heads
 * of the group (each row is read once for the whole group).
 * sel_count has the matching [batch][heads] shape; ids must be < seq_lens[b]
 * (others are skipped and flagged).  probs (optional): device fp32
 * [batch][H_q][sel_cap], the softmax probability of every listed token, in
 * list order (a second, short launch normalizes them).  An empty list gives 0.
 * ws: kv_sparse_attn_ws(layout, seqs, sel_cap) bytes.
 * ---------------------------------------------------------------------- */
int kv_sparse_attn(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                   const uint16_t* q, const int32_t* sel, int32_t sel_cap,
                   const int32_t* sel_count, int32_t sel_per_kv_head,
                   float* out, float* probs,
                   void* ws, size_t ws_bytes, void* stream);
size_t kv_sparse_attn_ws(const kvq_layout* layout, const kvq_seqs* seqs, int32_t sel_cap);

/* ------------------------------------------------------------------------
 * Fused decode step of a sparse (fp16) layer, two launches instead of four:
 *
 * kv_append_critical_score = kv_page_append (fp16 layer) + kv_critical_score.
 * The newest token (position seq_lens[b] - 1, rows k_new/v_new as in
 * kv_page_append) is written to k16/v16, kT and k_absmax, and the scores of
 * every token -- the newest included -- are those kv_critical_score would
 * give after the append.  If hist is not NULL (device uint32
 * [batch][H_q][4096], zero-filled before first use), the call adds the
 * histogram of bits 31..20 of the order-preserving keys of the candidate
 * scores (positions n_sink <= t < T - window) for kv_select_sparse_attn,
 * which clears it again.  ws: kv_append_critical_score_ws() bytes.
 *
 * kv_select_sparse_attn = kv_topk_select + kv_sparse_attn with one list per
 * q head: the selection of kv_topk_select (same k_fixed / ratio / n_sink /
 * window) and exact attention over it, in one launch; the output is that of
 * kv_sparse_attn on the selected list.  hist: NULL or the histogram written
 * by kv_append_critical_score for these scores with the same n_sink, window
 * and seq_lens.  sel / sel_count: optional (NULL) copies of the selection in
 * kv_topk_select's layout.  T <= 360448.  ws: kv_select_sparse_attn_ws().
 * ---------------------------------------------------------------------- */
int kv_append_critical_score(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                             const uint16_t* k_new, const uint16_t* v_new, const uint16_t* q,
                             int32_t n_crit, int32_t* crit, float* scores, int64_t score_stride,
                             uint32_t* hist, int32_t n_sink, int32_t window,
                             void* ws, size_t ws_bytes, void* stream);
size_t kv_append_critical_score_ws(void);

int kv_select_sparse_attn(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                          const uint16_t* q, const float* scores, int64_t score_stride, uint32_t* hist,
                          int32_t k_fixed, double ratio, int32_t n_sink, int32_t window,
                          int32_t* sel, int32_t sel_cap, int32_t* sel_count, float* out,
                          void* ws, size_t ws_bytes, void* stream);
size_t kv_select_sparse_attn_ws(void);

/* ------------------------------------------------------------------------
 * kv_sparse_layer_decode -- the whole decode step of a sparse (fp16) layer in
 * one launch: kv_page_append of the newest token, kv_critical_score,
 * kv_topk_select and kv_sparse_attn (one list per q head).  Equal results:
 * the same appended rows, the same fp32 scores and selection, the attention
 * of kv_sparse_attn over that selection [TailorKV §2.3; KVSurvey §三.1;
 * Meeting §3.2].  The scores never leave the GPU's shared memory unless
 * `scores` (optional, device fp32 [batch][H_q][score_stride]) asks for a
 * copy; `sel`/`sel_count` (optional) receive the selection as
 * kv_topk_select writes it.  T <= 360448.  q, k_new and v_new 16-byte
 * aligned; the newest token's row is attended from k_new/v_new, so no CTA
 * depends on another cluster's append.  ws: kv_sparse_layer_decode_ws().
 * ---------------------------------------------------------------------- */
int kv_sparse_layer_decode(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                           const uint16_t* k_new, const uint16_t* v_new, const uint16_t* q, int32_t n_crit,
                           int32_t k_fixed, double ratio, int32_t n_sink, int32_t window,
                           float* scores, int64_t score_stride,
                           int32_t* sel, int32_t sel_cap, int32_t* sel_count, float* out,
                           void* ws, size_t ws_bytes, void* stream);
size_t kv_sparse_layer_decode_ws(void);

/* ------------------------------------------------------------------------
 * kv_mixed_layer_decode -- kv_sparse_layer_decode for a layer whose heads were
 * classified one by one [TailorKV §6: the layer-level strategy carried down to
 * attention heads; §2.1 dense-preference score]: every (sequence, q head) is
 * dispatched on the device by its kv head's class, dense[b][g] (device int32
 * [batch][H_kv], e.g. from kvq_classify_heads): non-zero -> the head attends
 * every cached token exactly (no critical scores, no selection; a `sel` copy
 * lists every token); zero -> the sparse path of kv_sparse_layer_decode
 * (critical scores, top-K with sinks and window, attention over the
 * selection).  The newest token is appended for every kv head.  Two launches,
 * stream-ordered: the cluster launch of kv_sparse_layer_decode, in which a
 * dense head's clusters only append and list; then the dense kv heads'
 * attention, the GQ q heads of a kv head sharing every staged K/V tile on the
 * tensor cores (the CTAs of sparse kv heads return at once).  Other arguments
 * as kv_sparse_layer_decode (no score copy).
 * ws: kv_mixed_layer_decode_ws(layout, seqs) bytes.
 * ---------------------------------------------------------------------- */
int kv_mixed_layer_decode(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                          const uint16_t* k_new, const uint16_t* v_new, const uint16_t* q, int32_t n_crit,
                          int32_t k_fixed, double ratio, int32_t n_sink, int32_t window,
                          const int32_t* dense, int32_t* sel, int32_t sel_cap, int32_t* sel_count,
                          float* out, void* ws, size_t ws_bytes, void* stream);
size_t kv_mixed_layer_decode_ws(const kvq_layout* layout, const kvq_seqs* seqs);

/* Head-level classification [TailorKV §6, §2.1], host code: kv head g (of
 * n_kv_heads; its q heads g*G .. g*G+G-1, G = n_q_heads / n_kv_heads) is dense
 * (quantization-friendly) when (sum over its q heads, ascending, of P[h]) / G /
 * n_q > tau, in double.  P: host fp32 [n_q_heads] dense-preference scores
 * (kv_dense_pref_score of one sequence); dense: host int32 [n_kv_heads] out
 * (1 dense, 0 sparse).  Returns the number of dense kv heads, or a negative
 * error.  With one kv head this is the layer rule (mean_h P_h / n_q > tau). */
int kvq_classify_heads(const float* P, int32_t n_q_heads, int32_t n_kv_heads, int32_t n_q, double tau,
                       int32_t* dense);

/* ------------------------------------------------------------------------
 * a7: kv_h2o_accumulate -- H2O heavy-hitter bookkeeping [KVSurvey §三.2, §三.1].
 *
 * Per (sequence b, kv head g) a retained list (unordered) of token positions
 * retained[b][g][0..n) with cumulative scores cum[b][g][0..n), n =
 * retained_count[b][g] <= cap.  probs: device fp32 [batch][H_q][cap] from
 * kv_sparse_attn with sel_per_kv_head == 1 on that list.
 *   1. cum[i] += p_0[i] + p_1[i] + ... (the group's heads summed in ascending
 *      order in fp32, then added to cum).
 *   2. With T = seq_lens[b], protected tokens are sinks (pos < n_sink) and
 *      the next step's window (pos >= T + 1 - window).  Unprotected tokens
 *      are evicted, lowest (cum, position) first, until n <= budget - 1 when
 *      new_pos is given, else n <= budget.
 *   3. If new_pos (device int32 [batch], may be NULL) has new_pos[b] >= 0,
 *      that position is appended with cum 0.
 * Eviction keeps the list order except that a single eviction moves the last
 * entry into the freed slot.  n_evicted (optional): device int32
 * [batch][H_kv], evictions of this call.
 * ws: kv_h2o_accumulate_ws() bytes (status word only).
 * ---------------------------------------------------------------------- */
int kv_h2o_accumulate(const kvq_layout* layout, const kvq_seqs* seqs,
                      const float* probs, int32_t* retained, int32_t* retained_count,
                      float* cum, int32_t cap, int32_t budget, int32_t n_sink, int32_t window,
                      const int32_t* new_pos, int32_t* n_evicted,
                      void* ws, size_t ws_bytes, void* stream);
size_t kv_h2o_accumulate_ws(void);

/* ------------------------------------------------------------------------
 * a8: kv_dense_pref_score -- [TailorKV §2.1] P = n_q - sum over the n_q most
 * recent queries of the sum of the top-k entries of softmax(q K^T/sqrt(d)).
 * Query i sits at position T - n_q + i and sees keys 0..T-n_q+i (causal);
 * a row shorter than topk contributes all its entries.
 *
 * Reads fp16 keys k16 through the block table.  q_recent: device fp16
 * [batch][H_q][n_q][d], 16-byte aligned; P: device fp32 [batch][H_q].  The
 * layer is quantization-friendly when mean_h P/n_q > tau (decided by the
 * caller; kvq_classify_heads per kv head).  Two launches: the scores of the
 * GQ*n_q query rows of a kv head against its keys as tensor-core products
 * (fp16 inputs, exact products, fp32 sums; K read once per kv head) into the
 * workspace, then one CTA per query row for max, sum, the k-th largest score
 * (radix select) and the top-k mass; no length limit.  1 <= n_q <= T;
 * (n_q_heads / n_kv_heads) * n_q <= 512.
 * ws: kv_dense_pref_score_ws(layout, seqs, n_q) bytes, which includes the
 * score matrix: batch * H_q * n_q * ceil(max_len / 128) * 128 fp32
 * (512 MiB for one sequence of 32 q heads, n_q = 32, at 128K).
 * ---------------------------------------------------------------------- */
int kv_dense_pref_score(const kvq_layout* layout, const kvq_pool* pool, const kvq_seqs* seqs,
                        const uint16_t* q_recent, int32_t n_q, int32_t topk, float* P,
                        void* ws, size_t ws_bytes, void* stream);
size_t kv_dense_pref_score_ws(const kvq_layout* layout, const kvq_seqs* seqs, int32_t n_q);

/* ------------------------------------------------------------------------
 * a9: kv_offload_gather -- copy selected fp16 K and V rows of an offloaded
 * layer from host memory into an HBM staging buffer laid out as pages, so
 * that kv_sparse_attn can read it through an identity block table
 * [Meeting §4.2 double buffer; TailorKV §2.3, §3.1].
 *
 * src_k, src_v: mapped (or device) fp16 [n_heads][src_stride_h / d rows][d];
 * row t of head h is at src + h*src_stride_h + t*d.
 * sel: device int32 [batch=1][n_heads][sel_cap] ids, sel_count [n_heads].
 * dst_k, dst_v: device fp16 pages [ceil(sel_cap/16)][n_heads][16][d]; list
 * entry i of head h lands in page i/16, slot i%16.
 * ws: kv_offload_gather_ws() bytes (status word only).
 * ---------------------------------------------------------------------- */
int kv_offload_gather(const uint16_t* src_k, const uint16_t* src_v, int64_t src_stride_h,
                      int64_t src_rows, int32_t n_heads,
                      const int32_t* sel, int32_t sel_cap, const int32_t* sel_count,
                      uint16_t* dst_k, uint16_t* dst_v,
                      void* ws, size_t ws_bytes, void* stream);
size_t kv_offload_gather_ws(void);

/* ------------------------------------------------------------------------
 * Device helpers.
 * ---------------------------------------------------------------------- */

/* seq_lens[b] += delta for b < batch (device int32), on the stream. */
int kvq_seq_lens_add(int32_t* seq_lens, int32_t batch, int32_t delta, void* stream);

/* Copy-on-write support [KVSurvey §一.2]: copy every array of page src to
 * page dst (both in [0, num_blocks)) for the layer described by layout/pool. */
int kv_page_copy(const kvq_layout* layout, const kvq_pool* pool, int32_t src, int32_t dst,
                 void* stream);

/* Synchronizes the stream, reads and clears the status word of a workspace.
 * Returns KVQ_OK, KVQ_ERR_DEVICE_CHECK (with the failing check in
 * kvq_last_error) or KVQ_ERR_CUDA. */
int kvq_check(void* ws, void* stream);

/* Synchronizes the stream, copies the KVQ_N_PATH_COUNTERS diagnostic counters
 * of a workspace header to out[] (host) and clears them.  The counters tell
 * which code paths the kernels that used this workspace took (KVQ_PATH_*);
 * they never change a result. */
int kvq_read_path_counters(void* ws, uint32_t* out, void* stream);

/* Diagnostic (an addition of this library): launches one warp that runs the
 * bounded mbarrier wait the E4M3 attention uses for its bulk copies, on a
 * barrier that nothing completes.  The wait gives up after its poll limit
 * (a fraction of a second) and records a timeout in the workspace status
 * word, so the next kvq_check returns KVQ_ERR_DEVICE_CHECK ("a bounded wait
 * for an asynchronous copy gave up") and the context stays usable.  It shows
 * that a copy that never lands ends in a status, not a hang.
 * ws: at least 256 bytes, zeroed. */
int kvq_selftest_bounded_wait(void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Host page allocator [KVSurvey §一.1-§一.2]: free list of physical pages,
 * allocation on demand, reference counts for pages shared between sequences
 * (prefix sharing).  Pure host code; thread-compatible (one thread at a time
 * per allocator).
 * ---------------------------------------------------------------------- */
typedef struct kvq_allocator kvq_allocator;

/* seed == 0: pages handed out in ascending id order; otherwise in an order
 * shuffled by a splitmix64 sequence from `seed`. */
kvq_allocator* kvq_alloc_create(int64_t num_blocks, uint64_t seed);
void    kvq_alloc_destroy(kvq_allocator* a);
/* n pages with reference count 1 into ids[0..n); KVQ_ERR_NO_SPACE (nothing
 * taken) when fewer than n are free. */
int     kvq_block_alloc(kvq_allocator* a, int32_t n, int32_t* ids);
/* Add a reference (another sequence shares the page). */
int     kvq_block_ref(kvq_allocator* a, int32_t id);
/* Drop a reference; the page returns to the free list at zero. */
int     kvq_block_free(kvq_allocator* a, int32_t id);
/* Reference count of a page (0 = free), or a negative error. */
int     kvq_block_refcount(const kvq_allocator* a, int32_t id);
int64_t kvq_alloc_num_free(const kvq_allocator* a);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
