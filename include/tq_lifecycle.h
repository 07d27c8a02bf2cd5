/*
 * tq_lifecycle.h -- host-side lifecycle policy for the ternary weight copy.
 *
 * The decode path reads a second, ternary-packed copy of the FFN weights
 * (sparkinfer PR #1154, Summary).  That copy costs memory other work needs.
 * The review that rejected the first version of the copy (PR #1154, the
 * "long-context serving regression" closing comment) and the fix that
 * followed (PR #1160, commit message) ask for three things, which this
 * policy implements:
 *   1. At load, do not build the copy when the memory left after it could
 *      not hold the working set other work needs (known at startup).
 *   2. When any allocation fails while the copy is resident, release the
 *      copy and retry the allocation once (not only for one kind of
 *      allocation).
 *   3. Rebuild the copy once enough memory is free again, so one busy moment
 *      does not lose the copy for the rest of the process.
 *
 * The library allocates no device memory itself: every allocation, release,
 * free-memory query and copy build goes through caller-supplied hooks (with
 * PyTorch, torch.cuda allocations and torch.cuda.mem_get_info).  The policy
 * keeps all its state in the caller-owned tq_lifecycle struct; it calls no
 * CUDA function and is not thread-safe (one owner thread per struct).
 */
#ifndef TQ_LIFECYCLE_H
#define TQ_LIFECYCLE_H

#include <stddef.h>
#include <stdint.h>

#include "tq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* What an allocation is for (passed to the hooks). */
typedef enum { TQ_LC_COPY = 0, TQ_LC_OTHER = 1 } tq_lc_purpose;

/* State of the copy. */
typedef enum {
    TQ_LC_ABSENT = 0,   /* never built (before tq_lifecycle_load)                */
    TQ_LC_RESIDENT = 1, /* built; tq_lifecycle_copy() returns it                  */
    TQ_LC_SKIPPED = 2,  /* not built at load: too little memory for it + reserve  */
    TQ_LC_RELEASED = 3, /* released to let another allocation succeed             */
    TQ_LC_FAILED = 4    /* its allocation or build failed                         */
} tq_lc_state;

typedef struct {
    /* Allocate `bytes` of device memory; return NULL on failure (an
     * out-of-memory must not be raised through the hook). */
    void *(*alloc)(void *ctx, size_t bytes, int32_t purpose);
    /* Release memory that alloc returned. */
    void (*release)(void *ctx, void *ptr, size_t bytes, int32_t purpose);
    /* Device memory free now, in bytes. */
    size_t (*free_bytes)(void *ctx);
    /* Fill a freshly allocated copy (e.g. pack the weights into it); return 0
     * on success. */
    int32_t (*build)(void *ctx, void *copy, size_t bytes);
    void *ctx;
} tq_lifecycle_hooks;

typedef struct {
    size_t copy_bytes;      /* bytes of the copy (> 0)                                   */
    size_t reserve_bytes;   /* memory that must stay free after the copy is built        */
    size_t rebuild_margin;  /* extra free memory a rebuild needs beyond copy + reserve   */
    int32_t rebuild_after;  /* polls to wait after a release or failure before a rebuild */
} tq_lifecycle_config;

typedef struct {
    tq_lifecycle_config cfg;
    tq_lifecycle_hooks hooks;
    void *copy;                  /* the copy while resident, else NULL */
    int32_t state;               /* tq_lc_state */
    int32_t polls_since_change;  /* polls since the last release or failure */
    /* counters, for the caller's logs */
    int64_t builds;              /* successful builds, at load or later */
    int64_t rebuilds;            /* of which after a release, skip or failure */
    int64_t releases;            /* releases to let another allocation succeed */
    int64_t alloc_failures;      /* first attempts of other allocations that failed */
    int64_t retries_ok;          /* of which succeeded after the copy was released */
    int64_t build_failures;      /* copy allocations or builds that failed */
} tq_lifecycle;

/* Set up `lc` (no allocation).  TQ_ERR_INVALID_ARG: null pointers, a hook
 * missing, copy_bytes == 0 or rebuild_after < 0. */
tq_status tq_lifecycle_init(tq_lifecycle *lc, const tq_lifecycle_config *cfg, const tq_lifecycle_hooks *hooks);

/* Load-time decision (rule 1): builds the copy when free memory covers
 * copy_bytes + reserve_bytes, else leaves it SKIPPED.  Only from ABSENT;
 * returns TQ_OK whether or not it built (read lc->state), TQ_ERR_INVALID_ARG
 * for a null or already loaded lc. */
tq_status tq_lifecycle_load(tq_lifecycle *lc);

/* The copy while resident, else NULL: callers take the ternary path only
 * when this is non-NULL. */
void *tq_lifecycle_copy(const tq_lifecycle *lc);

/* Allocate memory for other work (rule 2): on failure with the copy
 * resident, release the copy and try once more.  NULL if it still fails. */
void *tq_lifecycle_alloc(tq_lifecycle *lc, size_t bytes, int32_t purpose);

/* Release memory tq_lifecycle_alloc returned. */
void tq_lifecycle_free(tq_lifecycle *lc, void *ptr, size_t bytes, int32_t purpose);

/* Rule 3, to be called between steps: once rebuild_after polls have passed
 * since the copy went away, rebuild it when free memory covers copy_bytes +
 * reserve_bytes + rebuild_margin.  Returns TQ_OK (read lc->state). */
tq_status tq_lifecycle_poll(tq_lifecycle *lc);

/* Release the copy now (e.g. before a known large allocation). */
void tq_lifecycle_release(tq_lifecycle *lc);

/* Release the copy if resident; lc may be reused after tq_lifecycle_init. */
void tq_lifecycle_destroy(tq_lifecycle *lc);

#ifdef __cplusplus
}
#endif

#endif /* TQ_LIFECYCLE_H */
