// seq.cuh -- device-side view of one (batch, head) sequence of a SeqArgs layout.
#pragma once

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

struct SeqView {
  int plane;  // plane of the tensors (b*H + h, or h with variable lengths)
  int start;  // first row of the sequence within the plane
  int len;    // rows (queries = keys) of the sequence; 0 if the offsets are invalid
};

// Sequence of flattened (batch, head) index bh. Variable-length offsets are
// checked (0 <= cu[b] <= cu[b+1] <= total, length <= N); a bad pair records
// kStatusBadSeqlens and yields an empty sequence, so nothing is read or
// written for it.
__device__ __forceinline__ SeqView seq_view(const SeqArgs& s, int bh, int* status) {
  SeqView v;
  if (s.cu_seqlens == nullptr) {
    v.plane = bh;
    v.start = 0;
    v.len = s.N;
    return v;
  }
  const int b = bh / s.H;
  v.plane = bh - b * s.H;
  const int c0 = __ldg(s.cu_seqlens + b), c1 = __ldg(s.cu_seqlens + b + 1);
  if (0 <= c0 && c0 <= c1 && c1 <= s.total && c1 - c0 <= s.N) {
    v.start = c0;
    v.len = c1 - c0;
  } else {
    report_status(status, kStatusBadSeqlens);
    v.start = 0;
    v.len = 0;
  }
  return v;
}

// Element offset of row `row` (within the sequence) of a plane.
__device__ __forceinline__ size_t seq_row_offset(const SeqArgs& s, const SeqView& v, int row) {
  return (size_t)v.plane * (size_t)s.plane_stride + (size_t)(v.start + row) * (size_t)s.row_stride;
}
// Index of row `row` in the per-row statistics (LSE).
__device__ __forceinline__ size_t seq_stat_index(const SeqArgs& s, const SeqView& v, int row) {
  return (size_t)v.plane * (size_t)s.stat_plane + (size_t)(v.start + row);
}

}  // namespace fa
