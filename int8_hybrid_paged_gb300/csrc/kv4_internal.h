// kv4_internal.h — host-side definitions shared by the C-ABI layer and the
// kernel launchers of libkv4. Not installed; include/kv4.h is the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kv4.h"

namespace kv4 {

constexpr int kHeadDim = 128;
constexpr int kPage = 16;
constexpr int kPageBlock = 2176;         // bytes per (page, KV head)
constexpr int kKCodeOff = 0;             // [16 tok][64 B]
constexpr int kVCodeOff = 1024;          // [64 dim pairs][16 tok]
constexpr int kKMetaOff = 2048;          // [16 tok] {fp16 delta, fp16 min}
constexpr int kVMetaOff = 2112;
constexpr int kMaxProtected = 256;       // s + w limit
constexpr int kDecodeThreads = 128;      // 4 warps per decode CTA
constexpr int kStages = 4;               // page stages per warp

// Device-resident decode plan, written by the plan kernel, read by split/merge.
struct PlanHeader {
    int32_t chunk_pages;   // INT4 pages per split work item
    int32_t total_items;   // work items of this call
    int32_t counter;       // dynamic work-fetch ticket
    int32_t pad;
};

struct AppendArgs {
    const uint16_t* k;            // [T][H][128] bf16 bits
    const uint16_t* v;
    const int32_t* cu_tokens;     // [n+1]
    const int32_t* slot_ids;      // [n]
    const int32_t* start_pos;     // [n]
    const int32_t* block_table;   // [n][stride]
    int32_t stride;
    int32_t n_seqs;
    int32_t total_tokens;
    int32_t num_heads;
    int32_t sink, window;
    int32_t max_slots;
    int64_t num_pages;
    uint8_t* pages;
    uint8_t* side;
    int64_t side_block_bytes;
    int32_t* seq_len;
    int32_t* err;
};

struct DecodeArgs {
    const uint16_t* q;            // [B][Hq][128] bf16 bits
    const int32_t* slot_ids;      // [B]
    const int32_t* context_lens;  // [B]
    const int32_t* block_table;   // [B][stride]
    int32_t stride;
    int32_t batch;
    int32_t num_q_heads;
    int32_t num_heads;            // H_kv
    int32_t group;                // G
    int32_t sink, window;
    int32_t max_slots;
    int64_t num_pages;
    float log2_scale;             // fl(sm_scale * log2 e)
    const uint8_t* pages;
    const uint8_t* side;
    int64_t side_block_bytes;
    const int32_t* seq_len;
    int32_t* err;
    // workspace
    PlanHeader* plan;
    int32_t* item_start;          // [B+1]
    float* part_o;                // [max_items][G][128]
    float2* part_ml;              // [max_items][G] {max (log2), sum}
    int32_t max_items;
    int32_t target_items;
    // outputs
    float* out;                   // [B][Hq][128]
    float* lse;                   // [B][Hq] or null
    // debug (any may be null)
    int8_t* dbg_q8;
    float* dbg_qscale;
    int32_t* dbg_qk;
    uint8_t* dbg_w;
    int32_t dbg_stride;
};

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);
// ev: null, or 4 events recorded before plan, between plan/split, split/merge, after merge.
cudaError_t launch_decode(const DecodeArgs& a, int grid, cudaStream_t stream, cudaEvent_t* ev);
// Persistent decode CTAs that fit on one SM (occupancy of the split kernel).
cudaError_t decode_ctas_per_sm(int group, int* ctas);

}  // namespace kv4
