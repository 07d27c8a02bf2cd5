// tq_lifecycle.cu -- host-side lifecycle policy of the ternary weight copy
// (include/tq_lifecycle.h).  Host code only: every allocation, release,
// free-memory query and build goes through the caller's hooks.
#include "tq_lifecycle.h"

namespace {

bool hooks_ok(const tq_lifecycle_hooks *h) {
    return h != nullptr && h->alloc != nullptr && h->release != nullptr && h->free_bytes != nullptr &&
           h->build != nullptr;
}

// Free memory covers `need` bytes (no overflow for any size_t inputs).
bool covers(size_t free_now, size_t a, size_t b, size_t c) {
    if (a > free_now) return false;
    free_now -= a;
    if (b > free_now) return false;
    free_now -= b;
    return c <= free_now;
}

// Allocate and build the copy; on any failure the state is FAILED and
// nothing stays allocated.
void build_copy(tq_lifecycle *lc) {
    const tq_lifecycle_hooks &h = lc->hooks;
    void *p = h.alloc(h.ctx, lc->cfg.copy_bytes, TQ_LC_COPY);
    if (p == nullptr) {
        ++lc->build_failures;
        lc->state = TQ_LC_FAILED;
        lc->polls_since_change = 0;
        return;
    }
    if (h.build(h.ctx, p, lc->cfg.copy_bytes) != 0) {
        h.release(h.ctx, p, lc->cfg.copy_bytes, TQ_LC_COPY);
        ++lc->build_failures;
        lc->state = TQ_LC_FAILED;
        lc->polls_since_change = 0;
        return;
    }
    if (lc->state != TQ_LC_ABSENT) ++lc->rebuilds;
    ++lc->builds;
    lc->copy = p;
    lc->state = TQ_LC_RESIDENT;
}

void release_copy(tq_lifecycle *lc) {
    if (lc->state != TQ_LC_RESIDENT) return;
    lc->hooks.release(lc->hooks.ctx, lc->copy, lc->cfg.copy_bytes, TQ_LC_COPY);
    lc->copy = nullptr;
    lc->state = TQ_LC_RELEASED;
    lc->polls_since_change = 0;
    ++lc->releases;
}

}  // namespace

extern "C" {

tq_status tq_lifecycle_init(tq_lifecycle *lc, const tq_lifecycle_config *cfg, const tq_lifecycle_hooks *hooks) {
    if (lc == nullptr || cfg == nullptr || !hooks_ok(hooks)) return TQ_ERR_INVALID_ARG;
    if (cfg->copy_bytes == 0 || cfg->rebuild_after < 0) return TQ_ERR_INVALID_ARG;
    *lc = tq_lifecycle{};
    lc->cfg = *cfg;
    lc->hooks = *hooks;
    lc->state = TQ_LC_ABSENT;
    return TQ_OK;
}

tq_status tq_lifecycle_load(tq_lifecycle *lc) {
    if (lc == nullptr || lc->state != TQ_LC_ABSENT) return TQ_ERR_INVALID_ARG;
    const size_t free_now = lc->hooks.free_bytes(lc->hooks.ctx);
    if (!covers(free_now, lc->cfg.copy_bytes, lc->cfg.reserve_bytes, 0)) {
        lc->state = TQ_LC_SKIPPED;
        lc->polls_since_change = 0;
        return TQ_OK;
    }
    build_copy(lc);
    return TQ_OK;
}

void *tq_lifecycle_copy(const tq_lifecycle *lc) {
    return lc != nullptr && lc->state == TQ_LC_RESIDENT ? lc->copy : nullptr;
}

void *tq_lifecycle_alloc(tq_lifecycle *lc, size_t bytes, int32_t purpose) {
    if (lc == nullptr) return nullptr;
    const tq_lifecycle_hooks &h = lc->hooks;
    void *p = h.alloc(h.ctx, bytes, purpose);
    if (p != nullptr) return p;
    ++lc->alloc_failures;
    if (lc->state != TQ_LC_RESIDENT) return nullptr;
    release_copy(lc);
    p = h.alloc(h.ctx, bytes, purpose);
    if (p != nullptr) ++lc->retries_ok;
    return p;
}

void tq_lifecycle_free(tq_lifecycle *lc, void *ptr, size_t bytes, int32_t purpose) {
    if (lc == nullptr || ptr == nullptr) return;
    lc->hooks.release(lc->hooks.ctx, ptr, bytes, purpose);
}

tq_status tq_lifecycle_poll(tq_lifecycle *lc) {
    if (lc == nullptr) return TQ_ERR_INVALID_ARG;
    if (lc->state == TQ_LC_RESIDENT || lc->state == TQ_LC_ABSENT) return TQ_OK;
    if (lc->polls_since_change < lc->cfg.rebuild_after) {
        ++lc->polls_since_change;
        return TQ_OK;
    }
    const size_t free_now = lc->hooks.free_bytes(lc->hooks.ctx);
    if (covers(free_now, lc->cfg.copy_bytes, lc->cfg.reserve_bytes, lc->cfg.rebuild_margin)) build_copy(lc);
    return TQ_OK;
}

void tq_lifecycle_release(tq_lifecycle *lc) {
    if (lc != nullptr) release_copy(lc);
}

void tq_lifecycle_destroy(tq_lifecycle *lc) {
    if (lc == nullptr) return;
    if (lc->state == TQ_LC_RESIDENT) {
        lc->hooks.release(lc->hooks.ctx, lc->copy, lc->cfg.copy_bytes, TQ_LC_COPY);
        lc->copy = nullptr;
    }
    lc->state = TQ_LC_ABSENT;
}

}  // extern "C"
