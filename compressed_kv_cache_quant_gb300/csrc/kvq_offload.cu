// a9 kv_offload_gather: copy the selected fp16 K/V rows of an offloaded layer
// from host memory (read directly by the GPU over the host link) into an HBM
// staging buffer laid out as pages [Meeting §4.2 double buffer; TailorKV
// §2.3 and §3.1 "critical token buffer", zero-copy mapping].
#include "kvq_internal.cuh"

namespace {

constexpr int D = KVQ_HEAD_DIM;
constexpr int PG = KVQ_BLOCK_TOKENS;
constexpr int GA_NT = 256;
constexpr int GA_ROWS = GA_NT / 16;  // one half-warp per row, 16 B per lane

struct GatherArgs {
    const uint16_t* src_k;
    const uint16_t* src_v;
    int64_t src_stride_h;
    int64_t src_rows;
    int32_t n_heads;
    const int32_t* sel;
    int32_t sel_cap;
    const int32_t* sel_count;
    uint16_t* dst_k;
    uint16_t* dst_v;
    KvqWsHeader* hdr;
};

__global__ void __launch_bounds__(GA_NT) gather_kernel(GatherArgs a) {
    const int h = blockIdx.y;
    const int i = blockIdx.x * GA_ROWS + (threadIdx.x >> 4);
    const int l16 = threadIdx.x & 15;
    const int n = min(a.sel_count[h], a.sel_cap);
    if (i >= n) return;
    const int32_t t = a.sel[(int64_t)h * a.sel_cap + i];
    if (t < 0 || t >= a.src_rows) {
        if (l16 == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_INDEX, t);
        return;
    }
    const int64_t so = (int64_t)h * a.src_stride_h + (int64_t)t * D + 8 * l16;
    const int64_t dof = (((int64_t)(i / PG) * a.n_heads + h) * PG + (i % PG)) * D + 8 * l16;
    const uint4 kx = *reinterpret_cast<const uint4*>(a.src_k + so);
    const uint4 vx = *reinterpret_cast<const uint4*>(a.src_v + so);
    *reinterpret_cast<uint4*>(a.dst_k + dof) = kx;
    *reinterpret_cast<uint4*>(a.dst_v + dof) = vx;
}

}  // namespace

extern "C" size_t kv_offload_gather_ws(void) { return sizeof(KvqWsHeader); }

extern "C" int kv_offload_gather(const uint16_t* src_k, const uint16_t* src_v, int64_t src_stride_h, int64_t src_rows,
                                 int32_t n_heads, const int32_t* sel, int32_t sel_cap, const int32_t* sel_count,
                                 uint16_t* dst_k, uint16_t* dst_v, void* ws, size_t ws_bytes, void* stream) {
    kvq_clear_error();
    int st = kvq_check_ws(ws, ws_bytes, kv_offload_gather_ws(), "kv_offload_gather");
    if (st) return st;
    KVQ_REQUIRE(src_k && src_v && sel && sel_count && dst_k && dst_v, KVQ_ERR_INVALID_ARG,
                "kv_offload_gather: NULL buffer");
    KVQ_REQUIRE(n_heads > 0 && sel_cap > 0 && src_rows >= 0 && src_stride_h >= src_rows * D && src_stride_h % 8 == 0,
                KVQ_ERR_INVALID_ARG, "kv_offload_gather: sizes (src_stride_h >= src_rows*128, multiple of 8)");
    KVQ_REQUIRE((((uintptr_t)src_k | (uintptr_t)src_v | (uintptr_t)dst_k | (uintptr_t)dst_v) & 15u) == 0,
                KVQ_ERR_INVALID_ARG, "kv_offload_gather: buffers must be 16-byte aligned");
    GatherArgs a;
    a.src_k = src_k;
    a.src_v = src_v;
    a.src_stride_h = src_stride_h;
    a.src_rows = src_rows;
    a.n_heads = n_heads;
    a.sel = sel;
    a.sel_cap = sel_cap;
    a.sel_count = sel_count;
    a.dst_k = dst_k;
    a.dst_v = dst_v;
    a.hdr = static_cast<KvqWsHeader*>(ws);
    dim3 grid((sel_cap + GA_ROWS - 1) / GA_ROWS, n_heads);
    gather_kernel<<<grid, GA_NT, 0, kvq_stream(stream)>>>(a);
    return kvq_launch_status("kv_offload_gather");
}
