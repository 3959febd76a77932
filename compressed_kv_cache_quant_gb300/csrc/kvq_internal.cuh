// Internal helpers shared by the libkvq translation units (not part of the ABI).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/kvq.h"

#define KVQ_ABI_VERSION 1

// ---------------------------------------------------------------- host side

// Records a thread-local error message and returns `code`.
int kvq_fail(int code, const char* fmt, ...);
// Clears the thread-local error text.
void kvq_clear_error();
// Number of SMs of the current device (cached per device); 152 when no device.
int kvq_num_sms();
// Maps a launch / runtime error of the last launch to KVQ_ERR_CUDA.
int kvq_launch_status(const char* what);

#define KVQ_REQUIRE(cond, code, ...)            \
    do {                                        \
        if (!(cond)) return kvq_fail((code), __VA_ARGS__); \
    } while (0)

static inline cudaStream_t kvq_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Workspace header: the first 256 bytes of every workspace.
struct KvqWsHeader {
    int32_t status;      // 0 = clean; otherwise the first failing check
    int32_t detail;      // an index describing the failure
    uint32_t path[KVQ_N_PATH_COUNTERS];  // diagnostics: how many CTAs took which code path
    int32_t pad[62 - KVQ_N_PATH_COUNTERS];
};
static_assert(sizeof(KvqWsHeader) == 256, "workspace header is 256 bytes");

// Device status codes written to KvqWsHeader::status.
enum KvqDeviceCheck : int32_t {
    KVQ_DEV_OK = 0,
    KVQ_DEV_BAD_PAGE = 1,       // block table entry outside [0, num_blocks)
    KVQ_DEV_BAD_INDEX = 2,      // selected / retained id outside [0, seq_len)
    KVQ_DEV_BAD_LENGTH = 3,     // seq_len outside [0, max_len] or capacity
    KVQ_DEV_OVERFLOW = 4,       // a list would exceed its capacity
    KVQ_DEV_RANGE = 5,          // a value beyond the fp16 range of a tensor-core operand
    KVQ_DEV_TIMEOUT = 6,        // a bounded wait for an asynchronous copy gave up
};

__host__ __device__ static inline size_t kvq_round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- device side

__device__ __forceinline__ void kvq_dev_flag(KvqWsHeader* h, int32_t code, int32_t detail) {
    if (h != nullptr && atomicCAS(&h->status, 0, code) == 0) h->detail = detail;
}

// Counts one use of code path `which` (KVQ_PATH_*) in the workspace header.
__device__ __forceinline__ void kvq_dev_count(KvqWsHeader* h, int which) {
    if (h != nullptr) atomicAdd(&h->path[which], 1u);
}

__device__ __forceinline__ float kvq_h2f(uint16_t x) { return __half2float(__ushort_as_half(x)); }
__device__ __forceinline__ uint16_t kvq_f2h(float x) { return __half_as_ushort(__float2half_rn(x)); }

// Order-preserving map of an fp32 value to uint32 (larger float -> larger key);
// -0 and +0 share one key.
__device__ __forceinline__ uint32_t kvq_float_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u << 1) == 0u) u = 0u;  // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Quantizer arithmetic, IEEE fp32 with explicit round-to-nearest operations:
// scale = (max - min) / (2^b - 1); code = clamp(rint((x - min) / scale), 0, 2^b - 1).
__device__ __forceinline__ float kvq_scale32(float mn, float mx, float levels) {
    return __fdiv_rn(__fsub_rn(mx, mn), levels);
}
__device__ __forceinline__ uint32_t kvq_code(float x, float mn, float scale32, float levels) {
    if (!(scale32 > 0.0f)) return 0u;
    float u = __fdiv_rn(__fsub_rn(x, mn), scale32);
    float r = rintf(u);
    r = fminf(fmaxf(r, 0.0f), levels);
    return (uint32_t)r;
}

// Symmetric code of x, stored offset by L: clamp(rint(fl(x / scale)), -L, L) + L; L for scale 0.
__device__ __forceinline__ uint32_t kvq_code_sym(float x, float scale32, int L) {
    if (!(scale32 > 0.0f)) return (uint32_t)L;
    const float r = fminf(fmaxf(rintf(__fdiv_rn(x, scale32)), (float)-L), (float)L);
    return (uint32_t)((int)r + L);
}
// The stored zero of a symmetric group: -L * fp16(scale), exact in fp32 (rounded to fp16 on store).
__device__ __forceinline__ float kvq_sym_zero(float scale32, int L) {
    return -(float)L * __half2float(__float2half_rn(scale32));
}

__device__ __forceinline__ float kvq_warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float kvq_warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Programmatic dependent launch: a kernel launched with kvq_launch_pdl may be
// scheduled while the previous kernel of the stream is still running.  It calls
// kvq_pdl_begin() before touching global memory: that waits until the previous
// grid has completed and its writes are visible, then lets the next kernel of
// the stream be scheduled in turn.
__device__ __forceinline__ void kvq_pdl_begin() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
static inline cudaError_t kvq_launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                         Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// log2(e) / sqrt(128): scores are kept in the log2 domain, p = exp2(s - m).
#define KVQ_SCORE_LOG2_SCALE 0.12751743074048468f

// ---- bit layout of the quantized codes (b = bits per code, 16 / b codes per 16-bit half word)
//
// Codes travel in pairs: the two codes of a pair sit at the same offset in the low and the
// high half of a 32-bit word, so one AND/OR turns a pair into two fp16 numbers 1024 + code
// (times a power of two) for the tensor-core fragments.
//
// K token row (4b words, one per token and kv head in its page): the pair of channels
// (2p, 2p + 1) with p = 8s + r + 4e (s < 8, r < 4, e < 2) is the m-th (m = 2s + e) pair of
// column r: word r*b + m / (16/b), offset (m % (16/b)) * b.
__host__ __device__ static inline void kvq_k_code_pos(int c, int bits, int* word, int* bit) {
    const int p = c >> 1, s = p >> 3, r = p & 3, e = (p >> 2) & 1;
    const int m = 2 * s + e, per = 16 / bits;
    *word = r * bits + m / per;
    *bit = (m % per) * bits + 16 * (c & 1);
}

// V page block (64b words per page and kv head): channel d = 16t + 8u + x (x < 8, u < 2) and the
// token pair (2y, 2y + 1) of the page with y = r + 4e form the m-th (m = 4r + 2e + u) pair of row
// 8t + x: word (8t + x)*b + m / (16/b), offset (m % (16/b)) * b; the odd token in the high half.
__host__ __device__ static inline void kvq_v_code_pos(int tok, int d, int bits, int* word, int* bit) {
    const int t = d >> 4, x = d & 7, u = (d >> 3) & 1;
    const int y = tok >> 1, r = y & 3, e = y >> 2;
    const int m = 4 * r + 2 * e + u, per = 16 / bits;
    *word = (8 * t + x) * bits + m / per;
    *bit = (m % per) * bits + 16 * (tok & 1);
}

// Once per (kernel, device): prefer the largest shared-memory carveout, so that
// the kernels of a decode step never make the SMs repartition L1 and shared
// memory between launches, and allow `dyn_smem_max` bytes of dynamic shared
// memory.  Returns KVQ_OK or KVQ_ERR_CUDA.
int kvq_prepare_kernel(const void* func, int dyn_smem_max);
// kv_mixed_layer_decode's second launch (kvq_sparse.cu): the dense kv heads' attention over every token
size_t kvq_dense_heads_attn_ws(const kvq_layout* L, const kvq_seqs* S);
int kvq_dense_heads_attn(const kvq_layout* L, const kvq_pool* P, const kvq_seqs* S, const uint16_t* q,
                         const int32_t* dense, float* out, void* ws, cudaStream_t s);

// The code width of a layout (its bits without the KVQ_V_SYMMETRIC flag) and the flag.
static inline int kvq_code_bits(const kvq_layout* L) { return L->bits & 0xFF; }
static inline bool kvq_v_sym(const kvq_layout* L) { return (L->bits & KVQ_V_SYMMETRIC) != 0; }

// Validates the fields of a layout shared by all calls.  need_q: the call
// reads query heads (H_q / H_kv must be 1, 2, 4 or 8).
int kvq_check_layout(const kvq_layout* L, const char* fn, bool need_q);
// Validates the batch descriptor (pointers, sizes).
int kvq_check_seqs(const kvq_seqs* S, const char* fn);
// Validates only the sizes of a batch descriptor (for workspace queries).
int kvq_check_seqs_sizes(const kvq_seqs* S, const char* fn);
// Validates a workspace pointer / size pair against the required size.
int kvq_check_ws(void* ws, size_t ws_bytes, size_t need, const char* fn);
