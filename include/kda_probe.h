/*
 * kda_probe.h -- measurement probe of the KDA step's memory traffic
 * (libkda_probe_gb300.so; a bench instrument, not part of the step's API in
 * kda.h).  Return codes and device error flags are kda.h's.
 */
#ifndef KDA_PROBE_GB300_H
#define KDA_PROBE_GB300_H

#include <stdint.h>

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Measurement probe: the step's HBM page traffic without its arithmetic.
 * For every (request r, head h) item (item n = h * batch + r, the step's
 * order) the 64 KiB FP32 page the step reads is read into shared memory by
 * one TMA bulk copy and written by bulk stores to every page the step
 * writes: tokens == 1 (decode) reads state[slots[r], h] and writes it back
 * in place; tokens T > 1 (verify) reads state[slots[r, accepted[r]-1], h]
 * and writes it to state[slots[r, t], h] for each t < T whose slot is > 0.
 * One CTA per SM over contiguous item ranges (and, with `sched`, the
 * step's shared items) with a ring of `stages` (2 or 3) pages, as the step
 * schedules its pages.  Decode leaves the pool's
 * values unchanged.  Its bandwidth bounds what the step's page traffic can
 * reach.
 *   state     float [num_slots, heads, 128, 128], 16-byte aligned, in/out
 *   slots     int32 [batch, slot_cols] (device); a read slot <= 0 skips the
 *             item; any slot >= num_slots skips it and sets KDA_DEVERR_SLOT
 *   accepted  int32 [batch] (device, tokens > 1); outside 1..T skips the
 *             item and sets KDA_DEVERR_ACCEPTED
 *   err       optional device word (4-byte aligned) for KDA_DEVERR_* flags
 * Errors: KDA_ERR_NULL_ARGS, KDA_ERR_TOKENS (tokens outside 1..8),
 * KDA_ERR_SHAPE (negative sizes, num_slots < 1, stages outside 2..3,
 * slot_cols < 1, or slot_cols < tokens when tokens > 1),
 * KDA_ERR_NULL_POINTER, KDA_ERR_ALIGNMENT, KDA_ERR_DEVICE, KDA_ERR_LAUNCH;
 * nothing is launched on error.  One kernel on `stream`. */
typedef struct kda_probe_args {
  int32_t batch, heads, num_slots, stages;
  float *state;
  const int32_t *slots;
  int32_t *err;
  int32_t tokens, slot_cols;  /* 1 and 1 for decode                         */
  const int32_t *accepted;    /* tokens > 1 only                             */
  int32_t *sched;             /* optional i32 [2] scheduler words, as in     */
                              /* kda_args: the step's split between ranges   */
                              /* and shared items; NULL = ranges only        */
} kda_probe_args;
int kda_probe_page_copy(const kda_probe_args *args, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_PROBE_GB300_H */
