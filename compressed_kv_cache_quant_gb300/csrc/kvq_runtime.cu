// libkvq runtime: error reporting, device helpers, workspace status check and
// the host page allocator (free list + reference counts for shared pages).
#include <stdarg.h>
#include <stddef.h>
#include <stdio.h>
#include <string.h>

#include <map>
#include <mutex>
#include <vector>

#include "kvq_internal.cuh"

// ---------------------------------------------------------------- errors

static thread_local char g_err[512] = {0};

int kvq_fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

void kvq_clear_error() { g_err[0] = 0; }

extern "C" const char* kvq_last_error(void) { return g_err; }
extern "C" int kvq_version(void) { return KVQ_ABI_VERSION; }

int kvq_num_sms() {
    static std::mutex mu;
    static std::vector<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 152;
    }
    std::lock_guard<std::mutex> lk(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 152;
        }
        cache[dev] = n;
    }
    return cache[dev];
}

int kvq_prepare_kernel(const void* func, int dyn_smem_max) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> done;  // (kernel, device) -> dynamic limit set
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return kvq_fail(KVQ_ERR_CUDA, "no CUDA device");
    }
    std::lock_guard<std::mutex> lk(mu);
    auto it = done.find({func, dev});
    if (it != done.end() && it->second >= dyn_smem_max) return KVQ_OK;
    cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess && dyn_smem_max > 0)  // (static shared memory counts against the default 48 KB too)
        e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem_max);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kernel attributes: %s", cudaGetErrorString(e));
    done[{func, dev}] = dyn_smem_max;
    return KVQ_OK;
}

int kvq_launch_status(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return KVQ_OK;
}

// ---------------------------------------------------------------- device helpers

__global__ void kvq_seq_lens_add_kernel(int32_t* lens, int32_t n, int32_t delta) {
    kvq_pdl_begin();
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) lens[i] += delta;
}

extern "C" int kvq_seq_lens_add(int32_t* seq_lens, int32_t batch, int32_t delta, void* stream) {
    kvq_clear_error();
    KVQ_REQUIRE(seq_lens != nullptr && batch >= 0, KVQ_ERR_INVALID_ARG, "kvq_seq_lens_add: bad arguments");
    if (batch == 0) return KVQ_OK;
    int st = kvq_prepare_kernel((const void*)kvq_seq_lens_add_kernel, 0);
    if (st) return st;
    const cudaError_t e =
        kvq_launch_pdl(kvq_seq_lens_add_kernel, dim3((batch + 255) / 256), dim3(256), 0, kvq_stream(stream), seq_lens,
                       batch, delta);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kvq_seq_lens_add: %s", cudaGetErrorString(e));
    return KVQ_OK;
}

extern "C" int kv_page_copy(const kvq_layout* L, const kvq_pool* P, int32_t src, int32_t dst, void* stream) {
    kvq_clear_error();
    KVQ_REQUIRE(L && P, KVQ_ERR_INVALID_ARG, "kv_page_copy: NULL descriptor");
    KVQ_REQUIRE(L->head_dim == KVQ_HEAD_DIM && L->block_tokens == KVQ_BLOCK_TOKENS, KVQ_ERR_UNSUPPORTED,
                "kv_page_copy: head_dim must be 128 and block_tokens 16");
    KVQ_REQUIRE(src >= 0 && dst >= 0 && src < P->num_blocks && dst < P->num_blocks, KVQ_ERR_INVALID_ARG,
                "kv_page_copy: page id out of range");
    KVQ_REQUIRE(L->n_kv_heads > 0, KVQ_ERR_INVALID_ARG, "kv_page_copy: n_kv_heads");
    cudaStream_t s = kvq_stream(stream);
    const size_t H = (size_t)L->n_kv_heads, d = KVQ_HEAD_DIM, B = KVQ_BLOCK_TOKENS;
    struct Arr { void* base; size_t bytes_per_page; };
    Arr arrs[6];
    int n = 0;
    KVQ_REQUIRE((L->bits & ~(0xFF | KVQ_V_SYMMETRIC)) == 0, KVQ_ERR_UNSUPPORTED, "kv_page_copy: bits");
    const int cb = kvq_code_bits(L);
    if (cb == 16) {
        KVQ_REQUIRE(P->k16 && P->v16, KVQ_ERR_INVALID_ARG, "kv_page_copy: k16/v16 NULL");
        arrs[n++] = {P->k16, H * B * d * 2};
        arrs[n++] = {P->v16, H * B * d * 2};
    } else if (cb == KVQ_BITS_E4M3) {
        KVQ_REQUIRE(P->k_codes && P->v_codes, KVQ_ERR_INVALID_ARG, "kv_page_copy: k_codes/v_codes NULL");
        arrs[n++] = {P->k_codes, H * B * d};
        arrs[n++] = {P->v_codes, H * B * d};
    } else {
        KVQ_REQUIRE(P->k_codes && P->v_codes && P->k_sz && P->v_sz, KVQ_ERR_INVALID_ARG,
                    "kv_page_copy: quantized arrays NULL");
        KVQ_REQUIRE(L->v_group_dims == 32 || L->v_group_dims == 64 || L->v_group_dims == 128,
                    KVQ_ERR_UNSUPPORTED, "kv_page_copy: v_group_dims");
        const size_t R = d * (size_t)cb / 8;
        arrs[n++] = {P->k_codes, H * B * R};
        arrs[n++] = {P->v_codes, H * B * R};
        arrs[n++] = {P->k_sz, H * d * 4};
        arrs[n++] = {P->v_sz, H * B * (d / L->v_group_dims) * 4};
    }
    for (int i = 0; i < n; ++i) {
        char* b = static_cast<char*>(arrs[i].base);
        cudaError_t e = cudaMemcpyAsync(b + (size_t)dst * arrs[i].bytes_per_page, b + (size_t)src * arrs[i].bytes_per_page,
                                        arrs[i].bytes_per_page, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kv_page_copy: %s", cudaGetErrorString(e));
    }
    return KVQ_OK;
}

extern "C" int kvq_check(void* ws, void* stream) {
    kvq_clear_error();
    KVQ_REQUIRE(ws != nullptr, KVQ_ERR_INVALID_ARG, "kvq_check: NULL workspace");
    cudaStream_t s = kvq_stream(stream);
    int32_t hdr[2] = {0, 0};
    cudaError_t e = cudaMemcpyAsync(hdr, ws, sizeof(hdr), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kvq_check: %s", cudaGetErrorString(e));
    if (hdr[0] != 0) {
        static const char* names[] = {"ok", "page id outside the pool", "token id outside the sequence",
                                      "sequence length outside its bounds", "list capacity exceeded",
                                      "an operand beyond the fp16 range (query times K scale, or a V scale)",
                                      "a bounded wait for an asynchronous copy gave up"};
        const char* nm = (hdr[0] > 0 && hdr[0] <= 6) ? names[hdr[0]] : "unknown";
        int32_t zero[2] = {0, 0};
        e = cudaMemcpyAsync(ws, zero, sizeof(zero), cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kvq_check: %s", cudaGetErrorString(e));
        return kvq_fail(KVQ_ERR_DEVICE_CHECK, "device check failed: %s (detail %d)", nm, hdr[1]);
    }
    return KVQ_OK;
}

extern "C" int kvq_read_path_counters(void* ws, uint32_t* out, void* stream) {
    kvq_clear_error();
    KVQ_REQUIRE(ws != nullptr && out != nullptr, KVQ_ERR_INVALID_ARG, "kvq_read_path_counters: NULL argument");
    cudaStream_t s = kvq_stream(stream);
    void* dev = static_cast<char*>(ws) + offsetof(KvqWsHeader, path);
    const size_t n = sizeof(uint32_t) * KVQ_N_PATH_COUNTERS;
    cudaError_t e = cudaMemcpyAsync(out, dev, n, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dev, 0, n, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return kvq_fail(KVQ_ERR_CUDA, "kvq_read_path_counters: %s", cudaGetErrorString(e));
    return KVQ_OK;
}

// ---------------------------------------------------------------- head-level classification

extern "C" int kvq_classify_heads(const float* P, int32_t n_q_heads, int32_t n_kv_heads, int32_t n_q, double tau,
                                  int32_t* dense) {
    kvq_clear_error();
    KVQ_REQUIRE(P && dense, KVQ_ERR_INVALID_ARG, "kvq_classify_heads: NULL P / dense");
    KVQ_REQUIRE(n_kv_heads > 0 && n_q_heads > 0 && n_q_heads % n_kv_heads == 0 && n_q > 0, KVQ_ERR_INVALID_ARG,
                "kvq_classify_heads: head counts / n_q");
    const int G = n_q_heads / n_kv_heads;
    int n_dense = 0;
    for (int g = 0; g < n_kv_heads; ++g) {
        double sum = 0.0;
        for (int j = 0; j < G; ++j) sum += (double)P[g * G + j];  // ascending head order
        dense[g] = (sum / G) / n_q > tau ? 1 : 0;
        n_dense += dense[g];
    }
    return n_dense;
}

// ---------------------------------------------------------------- host page allocator

struct kvq_allocator {
    std::vector<int32_t> free_list;   // stack; back() is handed out next
    std::vector<int32_t> refcount;    // 0 = free
};

static uint64_t splitmix64(uint64_t& s) {
    uint64_t z = (s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

extern "C" kvq_allocator* kvq_alloc_create(int64_t num_blocks, uint64_t seed) {
    kvq_clear_error();
    if (num_blocks <= 0 || num_blocks > INT32_MAX) {
        kvq_fail(KVQ_ERR_INVALID_ARG, "kvq_alloc_create: num_blocks out of range");
        return nullptr;
    }
    kvq_allocator* a = new kvq_allocator();
    a->refcount.assign((size_t)num_blocks, 0);
    a->free_list.resize((size_t)num_blocks);
    // back() is handed out first: store ids descending so allocation is ascending.
    for (int64_t i = 0; i < num_blocks; ++i) a->free_list[(size_t)i] = (int32_t)(num_blocks - 1 - i);
    if (seed != 0) {
        uint64_t s = seed;
        for (int64_t i = num_blocks - 1; i > 0; --i) {
            int64_t j = (int64_t)(splitmix64(s) % (uint64_t)(i + 1));
            std::swap(a->free_list[(size_t)i], a->free_list[(size_t)j]);
        }
    }
    return a;
}

extern "C" void kvq_alloc_destroy(kvq_allocator* a) { delete a; }

extern "C" int kvq_block_alloc(kvq_allocator* a, int32_t n, int32_t* ids) {
    kvq_clear_error();
    KVQ_REQUIRE(a && n >= 0 && (n == 0 || ids), KVQ_ERR_INVALID_ARG, "kvq_block_alloc: bad arguments");
    KVQ_REQUIRE((size_t)n <= a->free_list.size(), KVQ_ERR_NO_SPACE, "kvq_block_alloc: %d pages asked, %zu free", n,
                a->free_list.size());
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = a->free_list.back();
        a->free_list.pop_back();
        a->refcount[(size_t)id] = 1;
        ids[i] = id;
    }
    return KVQ_OK;
}

extern "C" int kvq_block_ref(kvq_allocator* a, int32_t id) {
    kvq_clear_error();
    KVQ_REQUIRE(a && id >= 0 && (size_t)id < a->refcount.size(), KVQ_ERR_INVALID_ARG, "kvq_block_ref: bad id %d", id);
    KVQ_REQUIRE(a->refcount[(size_t)id] > 0, KVQ_ERR_INVALID_ARG, "kvq_block_ref: page %d is free", id);
    a->refcount[(size_t)id] += 1;
    return KVQ_OK;
}

extern "C" int kvq_block_free(kvq_allocator* a, int32_t id) {
    kvq_clear_error();
    KVQ_REQUIRE(a && id >= 0 && (size_t)id < a->refcount.size(), KVQ_ERR_INVALID_ARG, "kvq_block_free: bad id %d", id);
    KVQ_REQUIRE(a->refcount[(size_t)id] > 0, KVQ_ERR_INVALID_ARG, "kvq_block_free: page %d already free", id);
    if (--a->refcount[(size_t)id] == 0) a->free_list.push_back(id);
    return KVQ_OK;
}

extern "C" int kvq_block_refcount(const kvq_allocator* a, int32_t id) {
    kvq_clear_error();
    KVQ_REQUIRE(a && id >= 0 && (size_t)id < a->refcount.size(), KVQ_ERR_INVALID_ARG, "kvq_block_refcount: bad id");
    return a->refcount[(size_t)id];
}

extern "C" int64_t kvq_alloc_num_free(const kvq_allocator* a) {
    if (!a) return KVQ_ERR_INVALID_ARG;
    return (int64_t)a->free_list.size();
}

// ---------------------------------------------------------------- validation

int kvq_check_layout(const kvq_layout* L, const char* fn, bool need_q) {
    KVQ_REQUIRE(L != nullptr, KVQ_ERR_INVALID_ARG, "%s: NULL layout", fn);
    KVQ_REQUIRE(L->head_dim == KVQ_HEAD_DIM, KVQ_ERR_UNSUPPORTED, "%s: head_dim %d (only 128)", fn, L->head_dim);
    KVQ_REQUIRE(L->block_tokens == KVQ_BLOCK_TOKENS, KVQ_ERR_UNSUPPORTED, "%s: block_tokens %d (only 16)", fn,
                L->block_tokens);
    KVQ_REQUIRE(L->n_kv_heads > 0 && L->n_q_heads > 0, KVQ_ERR_INVALID_ARG, "%s: head counts", fn);
    const int cb = kvq_code_bits(L);
    KVQ_REQUIRE((L->bits & ~(0xFF | KVQ_V_SYMMETRIC)) == 0 &&
                    (cb == 1 || cb == 2 || cb == 4 || cb == 8 || cb == 16 || cb == KVQ_BITS_E4M3),
                KVQ_ERR_UNSUPPORTED, "%s: bits %d (1, 2, 4, 8, 16 or KVQ_BITS_E4M3)", fn, L->bits);
    KVQ_REQUIRE(!kvq_v_sym(L) || cb == 2 || cb == 4 || cb == 8, KVQ_ERR_UNSUPPORTED,
                "%s: symmetric V needs 2, 4 or 8 bits", fn);
    if (cb != 16 && cb != KVQ_BITS_E4M3) {
        KVQ_REQUIRE(L->k_group_tokens == KVQ_K_GROUP_TOKENS, KVQ_ERR_UNSUPPORTED, "%s: k_group_tokens %d (only 64)",
                    fn, L->k_group_tokens);
        KVQ_REQUIRE(L->v_group_dims == 32 || L->v_group_dims == 64 || L->v_group_dims == 128, KVQ_ERR_UNSUPPORTED,
                    "%s: v_group_dims %d (32, 64 or 128)", fn, L->v_group_dims);
    }
    if (need_q) {
        KVQ_REQUIRE(L->n_q_heads % L->n_kv_heads == 0, KVQ_ERR_INVALID_ARG, "%s: H_q %% H_kv != 0", fn);
        int g = L->n_q_heads / L->n_kv_heads;
        KVQ_REQUIRE(g == 1 || g == 2 || g == 4 || g == 8, KVQ_ERR_UNSUPPORTED, "%s: H_q/H_kv = %d (1, 2, 4 or 8)", fn,
                    g);
    }
    return KVQ_OK;
}

int kvq_check_seqs(const kvq_seqs* S, const char* fn) {
    KVQ_REQUIRE(S != nullptr, KVQ_ERR_INVALID_ARG, "%s: NULL seqs", fn);
    KVQ_REQUIRE(S->batch >= 0 && S->max_blocks >= 0 && S->max_len >= 0, KVQ_ERR_INVALID_ARG, "%s: negative sizes",
                fn);
    KVQ_REQUIRE(S->batch == 0 || S->seq_lens != nullptr, KVQ_ERR_INVALID_ARG, "%s: NULL seq_lens", fn);
    KVQ_REQUIRE((int64_t)S->max_len <= (int64_t)S->max_blocks * KVQ_BLOCK_TOKENS, KVQ_ERR_INVALID_ARG,
                "%s: max_len %d exceeds 16 * max_blocks", fn, S->max_len);
    return KVQ_OK;
}

int kvq_check_seqs_sizes(const kvq_seqs* S, const char* fn) {
    KVQ_REQUIRE(S != nullptr, KVQ_ERR_INVALID_ARG, "%s: NULL seqs", fn);
    KVQ_REQUIRE(S->batch >= 0 && S->max_blocks >= 0 && S->max_len >= 0, KVQ_ERR_INVALID_ARG, "%s: negative sizes",
                fn);
    return KVQ_OK;
}

int kvq_check_ws(void* ws, size_t ws_bytes, size_t need, const char* fn) {
    KVQ_REQUIRE(ws != nullptr, KVQ_ERR_INVALID_ARG, "%s: NULL workspace", fn);
    KVQ_REQUIRE(((uintptr_t)ws & 255u) == 0, KVQ_ERR_INVALID_ARG, "%s: workspace not 256-byte aligned", fn);
    KVQ_REQUIRE(ws_bytes >= need, KVQ_ERR_INVALID_ARG, "%s: workspace %zu bytes, %zu needed", fn, ws_bytes, need);
    return KVQ_OK;
}
