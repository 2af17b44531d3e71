/*
 * peagle_train.h -- C ABI of P-EAGLE's long-context training index work on
 * one GB300 (sm_103a): the amortized attention mask and the sequence
 * partitioning of one long training sequence.
 *
 * Source: "P-EAGLE: Parallel-Drafting EAGLE with Scalable Training" (paper
 * summary page), section 3 (a sequence of n tokens is expanded to n x K
 * positions; conditional drop-token (COD) sampling keeps the later depths at
 * a geometric rate r), 3.1 "Amortized Mask Construction" and 3.2 "Sequence
 * Partitioning"; the ScienceStack page of the paper, Figures 3 and 4.
 *
 * Rows.  Row (p, d) is prediction depth d = 0..K-1 at token position
 * p = 0..n-1, stored position-major at index p * K + d.  Depth 0 is the
 * next-token row of position p; depth d >= 1 is the d-th MASK row of the
 * draft whose next-token row is (p - d, 0), and exists only for p >= d.
 *
 * Attention rule.  Row (p, d) attends the depth-0 rows q <= p - d and the
 * MASK rows (p - d + e, e) for 1 <= e <= d -- the positions 0..p that a
 * drafting row at position p sees at inference.  The rule depends on p - q
 * only, so the mask of an n-token sample is the top-left (n K) x (n K)
 * block of the mask of any longer sample (Figure 3).
 *
 * Conventions are those of peagle.h: caller-owned device memory unless a
 * parameter says "host", asynchronous on `stream`, host-checkable errors
 * returned before anything is launched.  No handle is needed.
 */
#ifndef PEAGLE_TRAIN_H_
#define PEAGLE_TRAIN_H_

#include <stdint.h>

#include "peagle.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PE_MASK_BOOL_U8 = 0,      /* 1 = may attend, 0 = may not */
  PE_MASK_ADDITIVE_BF16 = 1 /* bf16 0 = may attend, -inf = may not */
} pe_mask_type;

/* Build the mask once for the longest sequence ([paper] 3.1): rows and
 * columns are the n_max * K rows above; out is [n_max * K, ld] elements of
 * mask_type, row stride ld >= n_max * K, with ld * element size a multiple
 * of 16 bytes and out 16-byte aligned.  Columns past n_max * K, and every
 * entry of a row or column that does not exist (p < d), read "may not".
 * HBM-write bound: (n_max K) x ld elements are written once.
 * PE_ERR_INVALID_ARGUMENT for n_max < 1, K outside [1, 1024], a bad ld or
 * alignment, or an unknown mask_type. */
pe_status pe_train_build_mask(int32_t n_max, int32_t K, int32_t mask_type, void* out,
                              int64_t ld, void* stream);

/* The mask of an n-token sample as a view of the mask built for n_max
 * ([paper] 3.1: a constant-time slice, no copy, no launch): *view = mask,
 * *view_rows = n * K, *view_ld = ld (elements).  PE_ERR_INVALID_ARGUMENT
 * unless 1 <= n <= n_max. */
pe_status pe_train_mask_view(const void* mask, int64_t ld, int32_t n_max, int32_t K, int32_t n,
                             const void** view, int64_t* view_rows, int64_t* view_ld);

/* COD sampling and sequence partitioning of one n-token sample
 * ([paper] 3, 3.2).
 *
 * COD: depth 0 is kept whole; row (p, d >= 1) is kept when its dependency
 * (p - 1, d - 1) is kept and u[p * K + d] < r (u: [n, K] fp32 draws in
 * [0, 1) chosen by the caller; depth-0 entries are unused).
 * Partition into S segments, bounds (HOST, S + 1 entries) with
 * bounds[0] = 0 < bounds[1] < ... < bounds[S] = n, S <= 64: kept rows of
 * depths 0 and 1 belong to the segment whose range [bounds[s],
 * bounds[s + 1]) holds p; a deeper row belongs to its dependency's segment;
 * each segment also lists, as context, the depth-0 rows before bounds[s].
 *
 * Outputs (device): keep [n, K] (1 = kept), seg [n, K] (owning segment, -1
 * for dropped rows), offsets [S + 1] into rows / owned, rows (layout
 * indices p * K + d of each segment's rows, in increasing order: its
 * context rows, then its own) and owned (1 = own row, 0 = context).
 * counts [S] is scratch.  rows and owned hold `capacity` entries, which
 * must be at least bounds[0] + ... + bounds[S - 1] + n * K.
 * PE_ERR_INVALID_ARGUMENT for n < 1, K < 1, S outside [1, 64], bad bounds,
 * a null pointer or too small a capacity. */
pe_status pe_train_partition(int32_t n, int32_t K, float r, const float* u, int32_t S,
                             const int32_t* bounds, uint8_t* keep, int32_t* seg,
                             int32_t* counts, int32_t* offsets, int32_t* rows,
                             uint8_t* owned, int64_t capacity, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PEAGLE_TRAIN_H_ */
