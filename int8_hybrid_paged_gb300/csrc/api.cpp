// api.cpp — the C ABI of libkv4 (declared in include/kv4.h): argument
// validation, pool ownership, workspace sizing and kernel launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "kv4_internal.h"

struct kv4_cache {
    kv4_cache_config cfg;
    int device = 0;
    int num_sms = 0;
    int grid[5] = {0, 0, 0, 0, 0};        // persistent decode CTAs per group size (index G)
    uint8_t* pages = nullptr;
    size_t pages_bytes = 0;
    uint8_t* side = nullptr;
    size_t side_bytes = 0;
    size_t side_block = 0;
    int32_t* seq_len = nullptr;
    int32_t* err = nullptr;
    unsigned char* ws = nullptr;           // decode workspace (layout: decode_workspace_bytes)
    size_t ws_bytes = 0;
    int32_t max_group = 0;
    const float* rope = nullptr;           // RoPE table (kv4_cache_set_rope), or null
    int32_t rope_max_pos = 0;
    // profiling: 4 events per recorded decode call
    std::vector<cudaEvent_t> events;
    int prof_capacity = 0;
    int prof_calls = 0;
    bool profiling = false;
};

namespace {

bool group_supported(int g) { return g == 1 || g == 2 || g == 4; }

void drop_events(kv4_cache* c)
{
    for (cudaEvent_t e : c->events) cudaEventDestroy(e);
    c->events.clear();
    c->prof_capacity = 0;
    c->prof_calls = 0;
    c->profiling = false;
}

void release(kv4_cache* c)
{
    drop_events(c);
    cudaFree(c->pages);
    cudaFree(c->side);
    cudaFree(c->seq_len);
    cudaFree(c->err);
    cudaFree(c->ws);
}

template <typename T>
bool alloc_zero(T** p, size_t bytes)
{
    if (bytes == 0) bytes = 16;
    if (cudaMalloc(reinterpret_cast<void**>(p), bytes) != cudaSuccess) {
        *p = nullptr;
        return false;
    }
    return cudaMemset(*p, 0, bytes) == cudaSuccess;
}

kv4_status check_launch(cudaError_t e)
{
    return e == cudaSuccess ? KV4_OK : KV4_ERR_CUDA;
}

// Makes a cache's device current for one call and restores the caller's device after,
// so a call made with another device current still runs where the cache lives.
class DeviceScope {
  public:
    explicit DeviceScope(int dev)
    {
        ok_ = cudaGetDevice(&prev_) == cudaSuccess;
        if (ok_ && prev_ != dev) {
            ok_ = cudaSetDevice(dev) == cudaSuccess;
            switched_ = ok_;
        }
    }
    ~DeviceScope()
    {
        if (switched_) cudaSetDevice(prev_);
    }
    bool ok() const { return ok_; }

  private:
    int prev_ = 0;
    bool ok_ = false;
    bool switched_ = false;
};

}  // namespace

extern "C" {

const char* kv4_status_string(kv4_status s)
{
    switch (s) {
    case KV4_OK: return "ok";
    case KV4_ERR_INVALID_ARG: return "invalid argument";
    case KV4_ERR_UNSUPPORTED: return "unsupported configuration";
    case KV4_ERR_OUT_OF_MEMORY: return "out of device memory";
    case KV4_ERR_CUDA: return "CUDA runtime error";
    case KV4_ERR_OUT_OF_RANGE: return "size above the cache's configured limits";
    case KV4_ERR_DEVICE_FAULT: return "device-side index error (see kv4_get_device_error)";
    }
    return "unknown status";
}

kv4_status kv4_cache_create(const kv4_cache_config* cfg, kv4_cache** out)
{
    if (!cfg || !out) return KV4_ERR_INVALID_ARG;
    *out = nullptr;
    if (cfg->num_kv_heads < 1 || cfg->sink < 0 || cfg->window < 0 || cfg->num_pages < 1 ||
        cfg->max_slots < 1 || cfg->max_batch < 1 || cfg->max_q_heads < 1 || cfg->max_work_items < 0)
        return KV4_ERR_INVALID_ARG;
    if (cfg->head_dim != KV4_HEAD_DIM || cfg->page_size != KV4_PAGE_SIZE) return KV4_ERR_UNSUPPORTED;
    if (cfg->sink + cfg->window > kv4::kMaxProtected) return KV4_ERR_UNSUPPORTED;
    if (cfg->format < KV4_FORMAT_INT4_HYBRID || cfg->format > KV4_FORMAT_MXFP4) return KV4_ERR_INVALID_ARG;
    const bool kv8 = cfg->format == KV4_FORMAT_INT8, fp4 = cfg->format == KV4_FORMAT_NVFP4;
    const bool mx = cfg->format == KV4_FORMAT_MXFP4;
    if ((kv8 || fp4 || mx) && (cfg->sink != 0 || cfg->window != 0)) return KV4_ERR_INVALID_ARG;
    // the protected weights are formed per page: a page's protected positions must sit in
    // one side-buffer group of 16 rows, which s and w multiples of 16 guarantee
    if (cfg->sink % KV4_PAGE_SIZE != 0 || cfg->window % KV4_PAGE_SIZE != 0) return KV4_ERR_UNSUPPORTED;
    if (cfg->max_q_heads % cfg->num_kv_heads != 0) return KV4_ERR_INVALID_ARG;
    const int gmax = cfg->max_q_heads / cfg->num_kv_heads;
    if (gmax > 4) return KV4_ERR_UNSUPPORTED;
    if ((int64_t)cfg->num_pages * cfg->num_kv_heads > (int64_t)INT32_MAX * 8) return KV4_ERR_UNSUPPORTED;
    if (cfg->num_pages > INT32_MAX) return KV4_ERR_UNSUPPORTED;

    kv4_cache* c = new (std::nothrow) kv4_cache();
    if (!c) return KV4_ERR_OUT_OF_MEMORY;
    c->cfg = *cfg;
    c->max_group = gmax;
    if (cudaGetDevice(&c->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
        delete c;
        return KV4_ERR_CUDA;
    }
    for (int g = 1; g <= 4; g <<= 1) {
        int per_sm = 0;
        if (kv4::decode_ctas_per_sm(g, &per_sm) != cudaSuccess || per_sm < 1) per_sm = 1;
        c->grid[g] = c->num_sms * per_sm;
    }
    const int H = cfg->num_kv_heads;
    const int S = cfg->sink + cfg->window;
    c->side_block = (size_t)((S + 15) / 16) * kv4::kSideGroupBytes;
    c->pages_bytes = (size_t)cfg->num_pages * H *
                     (fp4 ? kv4::kPageBlock4f : kv8 ? kv4::kPageBlock8 : mx ? kv4::kPageBlockMx : kv4::kPageBlock);
    c->side_bytes = (size_t)cfg->max_slots * H * c->side_block;
    int grid_max = 0;
    for (int g = 1; g <= 4; g <<= 1) grid_max = std::max(grid_max, c->grid[g]);
    c->ws_bytes = kv4::decode_workspace_bytes(cfg->max_batch, cfg->max_q_heads, H, gmax, grid_max,
                                              nullptr, nullptr);
    bool ok = alloc_zero(&c->pages, c->pages_bytes) && alloc_zero(&c->side, c->side_bytes) &&
              alloc_zero(&c->seq_len, sizeof(int32_t) * cfg->max_slots) &&
              alloc_zero(&c->err, sizeof(int32_t)) && alloc_zero(&c->ws, c->ws_bytes);
    if (!ok || cudaDeviceSynchronize() != cudaSuccess) {
        release(c);
        delete c;
        cudaGetLastError();
        return KV4_ERR_OUT_OF_MEMORY;
    }
    *out = c;
    return KV4_OK;
}

kv4_status kv4_cache_free(kv4_cache* c)
{
    if (!c) return KV4_OK;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(c->device);
    cudaDeviceSynchronize();
    release(c);
    cudaSetDevice(prev);
    delete c;
    return KV4_OK;
}

kv4_status kv4_cache_get_info(const kv4_cache* c, kv4_cache_info* info)
{
    if (!c || !info) return KV4_ERR_INVALID_ARG;
    info->page_pool_dev = c->pages;
    info->page_pool_bytes = c->pages_bytes;
    info->side_pool_dev = c->side;
    info->side_pool_bytes = c->side_bytes;
    info->side_block_bytes = c->side_block;
    info->seq_len_dev = c->seq_len;
    info->num_sms = c->num_sms;
    info->decode_grid = c->grid[4];
    info->device = c->device;
    return KV4_OK;
}

kv4_status kv4_cache_set_rope(kv4_cache* c, const float* cos_sin, int max_pos)
{
    if (!c) return KV4_ERR_INVALID_ARG;
    if (!cos_sin) {
        c->rope = nullptr;
        c->rope_max_pos = 0;
        return KV4_OK;
    }
    if (max_pos < 1 || (reinterpret_cast<uintptr_t>(cos_sin) & 15)) return KV4_ERR_INVALID_ARG;
    c->rope = cos_sin;
    c->rope_max_pos = max_pos;
    return KV4_OK;
}

kv4_status kv4_append(kv4_cache* c, const void* k, const void* v, const int32_t* cu_tokens,
                      const int32_t* slot_ids, const int32_t* start_pos, const int32_t* block_table,
                      int stride, int n_seqs, int total_tokens, void* stream)
{
    if (!c || n_seqs < 0 || total_tokens < 0 || stride < 0) return KV4_ERR_INVALID_ARG;
    if (n_seqs == 0 || total_tokens == 0) return KV4_OK;
    if (!k || !v || !cu_tokens || !slot_ids || !start_pos || !block_table || stride < 1)
        return KV4_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 7) return KV4_ERR_INVALID_ARG;
    if ((int64_t)total_tokens * c->cfg.num_kv_heads > (int64_t)INT32_MAX * 8) return KV4_ERR_OUT_OF_RANGE;
    DeviceScope dev(c->device);
    if (!dev.ok()) return KV4_ERR_CUDA;
    kv4::AppendArgs a{};
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.cu_tokens = cu_tokens;
    a.slot_ids = slot_ids;
    a.start_pos = start_pos;
    a.block_table = block_table;
    a.stride = stride;
    a.n_seqs = n_seqs;
    a.total_tokens = total_tokens;
    a.num_heads = c->cfg.num_kv_heads;
    a.sink = c->cfg.sink;
    a.window = c->cfg.window;
    a.max_slots = c->cfg.max_slots;
    a.num_pages = c->cfg.num_pages;
    a.pages = c->pages;
    a.side = c->side;
    a.side_block_bytes = (int64_t)c->side_block;
    a.seq_len = c->seq_len;
    a.err = c->err;
    a.kv8 = c->cfg.format != KV4_FORMAT_INT4_HYBRID;
    a.fp4 = c->cfg.format == KV4_FORMAT_NVFP4;
    a.mx = c->cfg.format == KV4_FORMAT_MXFP4;
    a.rope = c->rope;
    a.rope_max_pos = c->rope_max_pos;
    return check_launch(kv4::launch_append(a, static_cast<cudaStream_t>(stream)));
}

static kv4_status decode_common(kv4_cache* c, const void* q, int num_q_heads,
                                const int32_t* slot_ids, const int32_t* context_lens,
                                const int32_t* block_table, int stride, int batch, float sm_scale,
                                float* out, float* lse, int8_t* dq8, float* dqs, int32_t* dqk,
                                uint8_t* dw, uint16_t* dp, int dbg_stride, void* stream)
{
    if (!c || batch < 0 || num_q_heads < 1 || stride < 0) return KV4_ERR_INVALID_ARG;
    if (batch == 0) return KV4_OK;
    if (!q || !slot_ids || !context_lens || !block_table || !out || stride < 1) return KV4_ERR_INVALID_ARG;
    if (!std::isfinite(sm_scale)) return KV4_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(q) & 7 || reinterpret_cast<uintptr_t>(out) & 15)
        return KV4_ERR_INVALID_ARG;
    const int H = c->cfg.num_kv_heads;
    if (num_q_heads % H != 0) return KV4_ERR_INVALID_ARG;
    const int G = num_q_heads / H;
    if (!group_supported(G)) return KV4_ERR_UNSUPPORTED;
    if (batch > c->cfg.max_batch || num_q_heads > c->cfg.max_q_heads) return KV4_ERR_OUT_OF_RANGE;
    if ((dqk || dw || dp) && dbg_stride < 1) return KV4_ERR_INVALID_ARG;
    DeviceScope dev(c->device);
    if (!dev.ok()) return KV4_ERR_CUDA;
    kv4::DecodeArgs a{};
    a.q = static_cast<const uint16_t*>(q);
    a.slot_ids = slot_ids;
    a.context_lens = context_lens;
    a.block_table = block_table;
    a.stride = stride;
    a.batch = batch;
    a.num_q_heads = num_q_heads;
    a.num_heads = H;
    a.group = G;
    a.sink = c->cfg.sink;
    a.window = c->cfg.window;
    a.max_slots = c->cfg.max_slots;
    a.num_pages = c->cfg.num_pages;
    a.log2_scale = (float)((double)sm_scale * 1.4426950408889634074);
    a.pages = c->pages;
    a.side = c->side;
    a.side_block_bytes = (int64_t)c->side_block;
    a.seq_len = c->seq_len;
    a.err = c->err;
    kv4::DecodeWorkspace ws{};
    kv4::decode_workspace_bytes(batch, num_q_heads, H, G, c->grid[G], &ws, c->ws);
    a.plan = ws.plan;
    a.cost_start = ws.cost_start;
    a.unit_seg = ws.unit_seg;
    a.qinfo = ws.qinfo;
    a.part_o = ws.part_o;
    a.part_ml = ws.part_ml;
    a.num_warps = c->grid[G] * (kv4::kDecodeThreads / 32);
    a.out = out;
    a.lse = lse;
    a.dbg_q8 = dq8;
    a.dbg_qscale = dqs;
    a.dbg_qk = dqk;
    a.dbg_w = dw;
    a.dbg_p = dp;
    a.dbg_stride = dbg_stride;
    a.kv8 = c->cfg.format != KV4_FORMAT_INT4_HYBRID;
    a.fp4 = c->cfg.format == KV4_FORMAT_NVFP4;
    a.mx = c->cfg.format == KV4_FORMAT_MXFP4;
    a.rope = c->rope;
    a.rope_max_pos = c->rope_max_pos;
    cudaEvent_t* ev = nullptr;
    if (c->profiling && c->prof_calls < c->prof_capacity) ev = &c->events[4 * c->prof_calls++];
    return check_launch(kv4::launch_decode(a, c->grid[G], static_cast<cudaStream_t>(stream), ev));
}

kv4_status kv4_decode_attention(kv4_cache* c, const void* q, int num_q_heads, const int32_t* slot_ids,
                                const int32_t* context_lens, const int32_t* block_table, int stride,
                                int batch, float sm_scale, float* out, float* lse, void* stream)
{
    return decode_common(c, q, num_q_heads, slot_ids, context_lens, block_table, stride, batch,
                         sm_scale, out, lse, nullptr, nullptr, nullptr, nullptr, nullptr, 0, stream);
}

kv4_status kv4_decode_attention_debug(kv4_cache* c, const void* q, int num_q_heads,
                                      const int32_t* slot_ids, const int32_t* context_lens,
                                      const int32_t* block_table, int stride, int batch,
                                      float sm_scale, float* out, float* lse, int8_t* q8,
                                      float* q_scale, int32_t* qk, uint8_t* w_hat, uint16_t* p_bits,
                                      int debug_stride, void* stream)
{
    return decode_common(c, q, num_q_heads, slot_ids, context_lens, block_table, stride, batch,
                         sm_scale, out, lse, q8, q_scale, qk, w_hat, p_bits, debug_stride, stream);
}

kv4_status kv4_profile_start(kv4_cache* c, int max_calls)
{
    if (!c || max_calls < 1) return KV4_ERR_INVALID_ARG;
    DeviceScope dev(c->device);
    if (!dev.ok()) return KV4_ERR_CUDA;
    drop_events(c);
    c->events.resize((size_t)4 * max_calls, nullptr);
    for (auto& e : c->events)
        if (cudaEventCreate(&e) != cudaSuccess) {
            e = nullptr;
            drop_events(c);
            return KV4_ERR_CUDA;
        }
    c->prof_capacity = max_calls;
    c->prof_calls = 0;
    c->profiling = true;
    return KV4_OK;
}

kv4_status kv4_profile_stop(kv4_cache* c, kv4_profile* out)
{
    if (!c || !out) return KV4_ERR_INVALID_ARG;
    *out = kv4_profile{0, 0.f, 0.f, 0.f};
    if (!c->profiling) return KV4_OK;
    DeviceScope dev(c->device);
    if (!dev.ok()) return KV4_ERR_CUDA;
    kv4_status st = KV4_OK;
    for (int i = 0; i < c->prof_calls; ++i) {
        cudaEvent_t* e = &c->events[4 * i];
        float t[3] = {0.f, 0.f, 0.f};
        if (cudaEventSynchronize(e[3]) != cudaSuccess) { st = KV4_ERR_CUDA; break; }
        for (int k = 0; k < 3; ++k)
            if (cudaEventElapsedTime(&t[k], e[k], e[k + 1]) != cudaSuccess) st = KV4_ERR_CUDA;
        out->plan_ms += t[0];
        out->split_ms += t[1];
        out->merge_ms += t[2];
        out->calls += 1;
    }
    drop_events(c);
    return st;
}

kv4_status kv4_qkv_append(kv4_cache* c, const void* x, const void* w, int num_q_heads, int d_model,
                          void* q_out, const int32_t* cu_tokens, const int32_t* slot_ids,
                          const int32_t* start_pos, const int32_t* block_table, int stride, int n_seqs,
                          int total_tokens, void* stream)
{
    if (!c || n_seqs < 0 || total_tokens < 0 || stride < 0 || num_q_heads < 1 || d_model < 64)
        return KV4_ERR_INVALID_ARG;
    if (n_seqs == 0 || total_tokens == 0) return KV4_OK;
    if (!x || !w || !q_out || !cu_tokens || !slot_ids || !start_pos || !block_table || stride < 1)
        return KV4_ERR_INVALID_ARG;
    if (d_model % 64 != 0 || (num_q_heads * KV4_HEAD_DIM) % 256 != 0) return KV4_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(q_out)) &
        15)
        return KV4_ERR_INVALID_ARG;
    if ((int64_t)total_tokens * c->cfg.num_kv_heads > (int64_t)INT32_MAX * 8) return KV4_ERR_OUT_OF_RANGE;
    DeviceScope dev(c->device);
    if (!dev.ok()) return KV4_ERR_CUDA;
    kv4::AppendArgs a{};
    a.cu_tokens = cu_tokens;
    a.slot_ids = slot_ids;
    a.start_pos = start_pos;
    a.block_table = block_table;
    a.stride = stride;
    a.n_seqs = n_seqs;
    a.total_tokens = total_tokens;
    a.num_heads = c->cfg.num_kv_heads;
    a.sink = c->cfg.sink;
    a.window = c->cfg.window;
    a.max_slots = c->cfg.max_slots;
    a.num_pages = c->cfg.num_pages;
    a.pages = c->pages;
    a.side = c->side;
    a.side_block_bytes = (int64_t)c->side_block;
    a.seq_len = c->seq_len;
    a.err = c->err;
    a.kv8 = c->cfg.format != KV4_FORMAT_INT4_HYBRID;
    a.fp4 = c->cfg.format == KV4_FORMAT_NVFP4;
    a.mx = c->cfg.format == KV4_FORMAT_MXFP4;
    a.rope = c->rope;
    a.rope_max_pos = c->rope_max_pos;
    return check_launch(
        kv4::launch_qkv_append(a, x, w, q_out, num_q_heads, d_model, static_cast<cudaStream_t>(stream)));
}

kv4_status kv4_linear_bf16(const void* x, const void* w, void* y, int M, int N, int K, int32_t* err,
                           void* stream)
{
    if (!x || !w || !y || M < 1 || N < 128 || K < 64 || N % 128 != 0 || K % 64 != 0)
        return KV4_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(y)) & 15)
        return KV4_ERR_INVALID_ARG;
    return check_launch(kv4::launch_linear_bf16(x, w, y, M, N, K, err, static_cast<cudaStream_t>(stream)));
}

kv4_status kv4_get_device_error(kv4_cache* c, int32_t* code, int clear)
{
    if (!code) return KV4_ERR_INVALID_ARG;
    if (!c) return kv4::noalloc_device_error(code, clear != 0) == cudaSuccess ? KV4_OK : KV4_ERR_CUDA;
    DeviceScope dev(c->device);
    if (!dev.ok()) return KV4_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return KV4_ERR_CUDA;
    if (cudaMemcpy(code, c->err, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return KV4_ERR_CUDA;
    if (clear && cudaMemset(c->err, 0, sizeof(int32_t)) != cudaSuccess) return KV4_ERR_CUDA;
    return KV4_OK;
}

}  // extern "C"
