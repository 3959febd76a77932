// a9 kv_offload_gather: copy the selected fp16 K/V rows of an offloaded layer
// from host memory (read directly by the GPU over the host link) into an HBM
// staging buffer laid out as pages [Meeting §4.2 double buffer; TailorKV
// §2.3 and §3.1 "critical token buffer", zero-copy mapping].
#include <algorithm>

#include "kvq_internal.cuh"

namespace {

constexpr int D = KVQ_HEAD_DIM;
constexpr int PG = KVQ_BLOCK_TOKENS;
constexpr int GA_NT = 512;
constexpr int GA_NHW = GA_NT / 16;  // half-warps per CTA: one row per half-warp, 16 B per lane
constexpr int GA_INFLIGHT = 4;      // rows in flight per half-warp

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

// A small persistent grid (a fraction of the SMs): the copy is bound by the host link's latency
// and bandwidth, not by SM work, so it keeps enough rows in flight with few CTAs and leaves the
// other SMs to kernels that run beside it (the attention of the previous layer).  Every
// half-warp walks the (head, list entry) slots with a grid stride, GA_INFLIGHT rows at a time.
__global__ void __launch_bounds__(GA_NT) gather_kernel(GatherArgs a) {
    const int l16 = threadIdx.x & 15;
    const int64_t stride = (int64_t)gridDim.x * GA_NHW;
    const int64_t total = (int64_t)a.n_heads * a.sel_cap;
    for (int64_t base = (int64_t)blockIdx.x * GA_NHW + (threadIdx.x >> 4); base < total;
         base += GA_INFLIGHT * stride) {
        uint4 kx[GA_INFLIGHT], vx[GA_INFLIGHT];
        int64_t dof[GA_INFLIGHT];
        bool ok[GA_INFLIGHT];
#pragma unroll
        for (int j = 0; j < GA_INFLIGHT; ++j) {
            const int64_t slot = base + j * stride;
            ok[j] = false;
            dof[j] = 0;
            if (slot >= total) continue;
            const int h = (int)(slot / a.sel_cap), i = (int)(slot % a.sel_cap);
            if (i >= min(a.sel_count[h], a.sel_cap)) continue;
            const int32_t t = a.sel[slot];
            if (t < 0 || t >= a.src_rows) {
                if (l16 == 0) kvq_dev_flag(a.hdr, KVQ_DEV_BAD_INDEX, t);
                continue;
            }
            const int64_t so = (int64_t)h * a.src_stride_h + (int64_t)t * D + 8 * l16;
            dof[j] = (((int64_t)(i / PG) * a.n_heads + h) * PG + (i % PG)) * D + 8 * l16;
            kx[j] = *reinterpret_cast<const uint4*>(a.src_k + so);
            vx[j] = *reinterpret_cast<const uint4*>(a.src_v + so);
            ok[j] = true;
        }
#pragma unroll
        for (int j = 0; j < GA_INFLIGHT; ++j) {
            if (!ok[j]) continue;
            *reinterpret_cast<uint4*>(a.dst_k + dof[j]) = kx[j];
            *reinterpret_cast<uint4*>(a.dst_v + dof[j]) = vx[j];
        }
    }
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
    const int64_t slots = (int64_t)n_heads * sel_cap;
    const int64_t want = (slots + GA_NHW * GA_INFLIGHT - 1) / (GA_NHW * GA_INFLIGHT);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, std::max(8, kvq_num_sms() / 4)));
    gather_kernel<<<grid, GA_NT, 0, kvq_stream(stream)>>>(a);
    return kvq_launch_status("kv_offload_gather");
}
