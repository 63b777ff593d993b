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
constexpr int kVCodeOff = 1024;          // [64 dim pairs][16 tok], fragment order
constexpr int kMetaOff = 2048;           // [8][K t, K t+8, V t, V t+8] {fp16 delta, fp16 min}
constexpr int kMaxProtected = 256;       // s + w limit
// Side buffer of one (slot, KV head): ceil((s+w)/16) groups of 16 rows, each two
// page-sized blocks laid out for the tensor-core fragments of the protected path:
//   K block: codes in two 1024-byte planes [16 rows][4 lanes][4 words], K meta
//            [8][row r, row r+8] at 2048
//   V block: codes [4][32 lanes][4 words] (PV A fragments), V meta [4][rows
//            t, t+8, t+4, t+12] at 2048
constexpr int kSideGroupBytes = 2 * kPageBlock;
constexpr int kSideKCodeOff = 0;
constexpr int kSideKMetaOff = 2048;
constexpr int kSideVCodeOff = kPageBlock;
constexpr int kSideVMetaOff = kPageBlock + 2048;
// A page block of the whole-cache 8-bit format: one side group, row r = token slot r.
constexpr int kPageBlock8 = kSideGroupBytes;
// A page block of the NVFP4 format: a K half and a V half of kFp4Half bytes each (codes
// in MMA-fragment order, E4M3 block scales, FP32 vector scales).
constexpr int kFp4Half = 1216;
constexpr int kPageBlock4f = 2 * kFp4Half;
constexpr int kFp4ScaleOff = 1024;
constexpr int kFp4GlobalOff = 1152;
// A page block of the MXFP4 format: a K half and a V half of kMxHalf bytes each (codes
// in the NVFP4 order, then the E8M0 scales of the four 32-value blocks of 16 tokens).
constexpr int kMxHalf = 1088;
constexpr int kPageBlockMx = 2 * kMxHalf;
constexpr int kMxScaleOff = 1024;
constexpr int kDecodeThreads = 512;      // 16 warps per decode CTA, one CTA per SM
constexpr int kStages = 5;               // page stages per warp
// The decode plan's cost line, in quarter-page units (fitted to measured per-warp times
// on the 8B-shaped and long-tail layers): an INT4 page costs 4, a protected stage item
// (half a side group, or half a page of a whole-cache format) 5. A (sequence, KV head)
// unit lays out as [kRunSetup][its INT4 pages][kProtSetup][its protected items]
// [kUnitFlush]: the gaps hold no items and stand for the setup of the INT4 run and of the
// protected run, and for the unit's flush, so that a span is charged for the runs it
// starts.
constexpr int kPageCost = 4;
constexpr int kProtCost = 5;
constexpr int kRunSetup = 12;
constexpr int kProtSetup = 16;
constexpr int kUnitFlush = 0;

// Device-resident decode plan, written by the prep kernel, read by split and merge.
struct PlanHeader {
    int32_t total_cost;    // stage items on the cost line
    int32_t span;          // cost per warp span
    int32_t total_items;   // partials of this call (protected units first, then span pieces)
    int32_t pad;
};

constexpr int kQInfoBytes = 144;   // per q head: 128 INT8 query bytes, {s_q, Σq8, QK offsets x2}

// Pointers into a decode workspace (cache-owned or the static no-allocation array).
struct DecodeWorkspace {
    PlanHeader* plan;
    int32_t* cost_start;   // [B+1]
    int32_t* unit_seg;     // [B*H+1] first partial of each (b, h) unit, then the total
    uint8_t* qinfo;        // [B*Hq][144]
    float2* part_ml;       // [items][G] {max (log2), normalizer}
    float* part_o;         // [items][G][128]
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
    int32_t kv8;                  // KV4_FORMAT_INT8 or NVFP4: the whole cache in pages, no side buffer
    int32_t fp4;                  // KV4_FORMAT_NVFP4: pages of kPageBlock4f bytes
    int32_t mx;                   // KV4_FORMAT_MXFP4: pages of kPageBlockMx bytes
    const float* rope;            // [rope_max_pos][128] cos | sin, or null (keys are post-RoPE)
    int32_t rope_max_pos;
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
    int32_t* cost_start;
    int32_t* unit_seg;
    uint8_t* qinfo;
    float* part_o;
    float2* part_ml;
    int32_t num_warps;            // warps of the persistent split grid
    // outputs
    float* out;                   // [B][Hq][128]
    float* lse;                   // [B][Hq] or null
    // debug (any may be null)
    int8_t* dbg_q8;
    float* dbg_qscale;
    int32_t* dbg_qk;
    uint8_t* dbg_w;
    uint16_t* dbg_p;              // bits of each protected position's PV weight
    int32_t dbg_stride;
    int32_t kv8;                  // KV4_FORMAT_INT8 or NVFP4: every position a row of a page group
    int32_t fp4;                  // KV4_FORMAT_NVFP4
    int32_t mx;                   // KV4_FORMAT_MXFP4
    const float* rope;            // [rope_max_pos][128] cos | sin, or null (queries are post-RoPE)
    int32_t rope_max_pos;
};

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);
// The projection X · W_qkvᵀ on the tcgen05 tensor cores with the append fused into its
// epilogue: Q columns to q_out (bf16), K and V columns appended as ap describes.
cudaError_t launch_qkv_append(const AppendArgs& ap, const void* x, const void* w, void* q_out, int num_q_heads,
                              int d_model, cudaStream_t stream);
// Y = X · Wᵀ (BF16 in and out, FP32 accumulation) on the tcgen05 tensor cores.
cudaError_t launch_linear_bf16(const void* x, const void* w, void* y, int M, int N, int K, int32_t* err,
                               cudaStream_t stream);
// ev: null, or 4 events recorded before plan, between plan/split, split/merge, after merge.
cudaError_t launch_decode(const DecodeArgs& a, int grid, cudaStream_t stream, cudaEvent_t* ev);
// Persistent decode CTAs that fit on one SM (occupancy of the split kernel); also
// opts the kernel in to its shared memory on the current device.
cudaError_t decode_ctas_per_sm(int group, int* ctas);
// Read (synchronously) and optionally clear the error word of the allocation-free decode
// on the current device.
cudaError_t noalloc_device_error(int32_t* code, bool clear);
// Bytes of a decode workspace for these sizes; with ws and base, also lays it out at base.
size_t decode_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int group, int grid,
                              DecodeWorkspace* ws, unsigned char* base);

}  // namespace kv4
