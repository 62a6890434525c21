// attention.h -- declarations shared by the host entry point (api.cu) and
// the decode-attention kernels (attention.cu).  Not part of the public ABI.
#pragma once

#include "internal.h"

namespace bi {

// Decode attention (attention.cu).
struct AttnParams {
  const void* q;               // [B, Hq, 128] bf16
  const int32_t* block_table;  // [B, bt_stride] page ids
  const int32_t* seq_lens;     // [B]
  uint32_t* ctl;               // [0] ticket counter, [1] items (both set by the plan kernel)
  uint32_t* items;             // (b << 16) | s of every (request, split) item
  float* part;                 // per (request, kv head, split): o^T [128][GP], m [GP], l [GP]
  int64_t bt_stride, num_pages;
  int64_t max_len;             // every seq_lens[b] must be in [0, max_len]
  int32_t Hq, Hkv, G, page_size, box_rows, split_size, n_split;
  int32_t page_shift, box_shift;  // log2 of page_size and of box_rows
  int32_t nreq;                   // requests (B)
  float qk_log2;               // scale * log2(e)
  int* status;                 // the device status word
};
struct AttnLaunch {
  CUtensorMap tmK, tmV;  // caches as [num_pages * page_size][2 Hkv][64], box {64, 2, box_rows},
                         // 128-byte swizzle (box_rows = min(page_size, 32))
  AttnParams p;
  void* out;             // [B, Hq, 128] bf16
  int64_t B;
  int32_t grid;          // stream kernel CTAs (one per SM)
  cudaStream_t stream;
};
// Calls with at most this many requests take their items from the lengths
// inside the stream kernel (no plan kernel).
constexpr int64_t kAttnStaticMaxB = 8;
cudaError_t launch_decode_attention(const AttnLaunch& A);

}  // namespace bi
