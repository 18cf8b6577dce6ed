// Bounds on the memory a matrix argument spans, checked before any plan is
// made: every product of extents, leading dimensions and strides taken later
// (in the planner, in byte offsets, in the kernels' 64-bit addressing) then
// stays far inside int64.
#pragma once

#include <stdint.h>

namespace dg {

// No operand may span more than 2^48 elements (at least 512 TB).
constexpr int64_t kMaxSpan = int64_t(1) << 48;

// True when `add` more elements, `count` times, still fit under kMaxSpan after
// `*span`; then adds them.  add and count are >= 0.
inline bool span_add(int64_t* span, int64_t add, int64_t count) {
    if (count <= 0 || add == 0) return true;
    if (add > kMaxSpan || count > kMaxSpan) return false;
    if (add > (kMaxSpan - *span) / count) return false;
    *span += add * count;
    return true;
}

// Span of an R x C matrix whose element (r, c) of batch entry b sits at
// b*bs + r*rs + c*cs (all strides >= 0), over `batch` entries.
inline bool strided_span_ok(int64_t R, int64_t C, int64_t rs, int64_t cs, int64_t batch,
                            int64_t bs) {
    int64_t span = 1;
    return span_add(&span, rs, R - 1) && span_add(&span, cs, C - 1) &&
           span_add(&span, bs, batch - 1);
}

// No operand may hold more than 2^56 elements over its batch, counted as
// logical elements (a broadcast or overlapping layout may reuse memory, but a
// dense workspace copy of the operand takes one slot per element).
constexpr int64_t kMaxCount = int64_t(1) << 56;

// batch * R * C <= kMaxCount, for non-negative factors.
inline bool count_ok(int64_t batch, int64_t R, int64_t C) {
    if (batch <= 0 || R <= 0 || C <= 0) return true;
    if (R > kMaxCount / batch) return false;
    const int64_t br = batch * R;
    return C <= kMaxCount / br;
}

}  // namespace dg
