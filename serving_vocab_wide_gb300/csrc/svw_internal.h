// svw_internal.h -- host-side declarations shared by the C-ABI layer and the
// kernel launchers.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/svw.h"

namespace svw {

// per-(row, chunk) partial result of the streaming row-statistics pass
struct alignas(16) Partial {
  float m;      // raw maximum of the chunk (argmax value in greedy mode)
  float s;      // sum of 2^((x - m) * log2(e)/T) over the chunk (unused when greedy)
  int32_t idx;  // argmax index (greedy), INT32_MAX if none
  int32_t nan;  // chunk holds a NaN (greedy)
};

// how one vocabulary row is split into work items
struct ChunkPlan {
  int32_t C;          // chunks per row (1..32)
  int32_t chunk_len;  // elements per chunk (multiple of 8)
};
ChunkPlan plan_chunks(int64_t V, int esize);

struct VerifyLayout {
  size_t part_off, counters_off, req_ok_off, global_ok_off, total;
};
VerifyLayout verify_layout(int32_t N, int64_t total_rows, int64_t V, int esize);

struct VerifyArgs {
  const void *target;
  const void *draft;
  int64_t V;
  int32_t N;
  const int32_t *cu;
  int64_t total_rows;
  int64_t rows_t;  // total_rows + N
  int32_t max_len;
  const int32_t *tokens;
  float k;  // log2(e) / T  (T > 0)
  uint64_t seed;
  int32_t *accept_len;
  int32_t *next_token;
  int32_t *status;
  Partial *part;
  int32_t *counters;
  int32_t *req_ok;
  int32_t *global_ok;
  int32_t C;
  int32_t chunk_len;
  int64_t total_items;
};

cudaError_t launch_verify(const VerifyArgs &a, int dtype, bool vec, bool greedy,
                          cudaStream_t stream);

struct OpdArgs {
  const void *target;
  const void *draft;
  int64_t V;
  int32_t N;
  const int32_t *cu;
  int64_t R;  // draft rows
  int32_t has_bonus;
  float k;     // log2(e) / T
  float invT;  // 1 / T
  float clip_c;
  float lambda_ce;
  float grad_scale;
  float *loss;
  float *dlogits;
  int32_t *status;
};

cudaError_t launch_opd(const OpdArgs &a, int dtype, bool bulk, cudaStream_t stream);

}  // namespace svw
