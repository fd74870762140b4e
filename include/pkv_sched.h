/*
 * pkv_sched.h -- host page allocator and page-budget admission for the
 * shared KV page pool (C ABI).
 *
 * "Hours of YouTube and 85 handtyped pages of notes on LLM Inference – Start
 * here" (the continuous-batching and page-pool items) describes the policy this
 * implements:
 *   - A request's admission budget is its largest processed prefix, prompt
 *     tokens + allowed new tokens - 1, rounded up to whole 16-token pages, in
 *     every layer. The allowed new tokens are clamped to the context limit
 *     (the last predicted token is returned, not processed again).
 *   - Budgets (credits) are separate from physical pages: a page is taken from
 *     the free list only when a sequence's KV length first reaches it, in each
 *     layer. Credits guarantee that growth never runs the pool dry.
 *   - Waiting requests are admitted in FIFO order when their budget fits next
 *     to the active ones (continuous batching), or, in static mode, only as a
 *     new group once every active request has finished. A request whose budget
 *     exceeds the whole pool is rejected at submission.
 *   - Finishing (at the budget, or early) returns the assigned pages and the
 *     unused credits.
 *   - Counters: pool size, peak active requests, largest decode batch, peak
 *     assigned pages, admission waits, free pages.
 *
 * All functions are host-only, not thread-safe per handle, and return 0 (or a
 * count) on success and a negative errno on failure: -EINVAL for bad
 * arguments or an unknown / inactive request, -ENOSPC for a request whose
 * budget exceeds the pool, -ENOMEM when the handle cannot be allocated.
 */
#ifndef PKV_SCHED_H
#define PKV_SCHED_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_sched pkv_sched_t;

typedef struct {
  int pool_pages;          /* pages in the pool */
  int free_pages;          /* pages on the free list now */
  int assigned_pages;      /* pages held by active requests now */
  int peak_assigned_pages; /* most pages held at once */
  int reserved_credits;    /* credits of the active requests now */
  int active;              /* active requests now */
  int waiting;             /* queued requests now */
  int peak_active;         /* most active requests at once */
  int largest_batch;       /* largest decode batch recorded by pkv_sched_note_batch */
  int admission_waits;     /* requests that had to wait for budget at least once */
  int admitted;            /* requests admitted so far */
  int completed;           /* requests finished so far */
  int rejected;            /* submissions rejected for exceeding the pool */
} pkv_sched_stats_t;

/*
 * New allocator over `num_pages` pages (ids 0 .. num_pages-1) for a model of
 * `num_layers` layers, 16-token pages and a context of `context_len` tokens.
 * static_batching != 0 selects static batching. The free list starts in a
 * seeded shuffled order (seed 0: ascending page ids).
 */
int pkv_sched_create(pkv_sched_t **out, int num_pages, int num_layers, int context_len,
                     int static_batching, uint64_t seed);
int pkv_sched_destroy(pkv_sched_t *s);

/*
 * Queue a request of prompt_len (>= 1, < context_len) tokens that may
 * generate up to max_new (>= 1) tokens, clamped to the context. Writes its id
 * (0, 1, 2, ... in submission order). -ENOSPC: its budget exceeds the pool
 * (the request is rejected, no id is written).
 */
int pkv_sched_submit(pkv_sched_t *s, int prompt_len, int max_new, int *request_id);

/* The credits (pages over all layers) a request of these sizes needs. */
int pkv_sched_budget(const pkv_sched_t *s, int prompt_len, int max_new);

/*
 * Admit waiting requests under the policy; writes up to max_ids admitted ids
 * in admission order and returns how many were admitted.
 */
int pkv_sched_admit(pkv_sched_t *s, int *ids, int max_ids);

/*
 * Make sure an active request has pages for kv_len tokens in every layer,
 * taking new pages from the free list (lazy assignment). -EINVAL if kv_len
 * exceeds the request's processed-prefix budget.
 */
int pkv_sched_grow(pkv_sched_t *s, int request_id, int kv_len);

/*
 * Copy a request's page ids for one layer into row[0 .. max_blocks-1],
 * padded with -1. Returns the number of pages assigned in that layer.
 */
int pkv_sched_block_row(const pkv_sched_t *s, int request_id, int layer, int32_t *row,
                        int max_blocks);

/* Finish an active request: its pages go back to the free list, its credits are released. */
int pkv_sched_finish(pkv_sched_t *s, int request_id);

/* Record the size of a decode batch (for the largest-batch counter). */
int pkv_sched_note_batch(pkv_sched_t *s, int batch);

int pkv_sched_stats(const pkv_sched_t *s, pkv_sched_stats_t *out);

#ifdef __cplusplus
}
#endif

#endif /* PKV_SCHED_H */
