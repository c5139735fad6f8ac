// Host-side pool for layout-coordinated parallel decoding (HPD-Parsing, part 2: shared-prefix KV reuse
// with context isolation; its scheduler forks a content branch at each <FORK> and frees the shared KV
// by reference count once every child is done).
//
// One shared prefix -- the context the layout (parent) branch has built so far -- grows by appending.
// A fork records the current prefix length as the child's fork position: the child sees exactly the
// prefix rows [0, fork position) without any copy.  Each child owns a fixed slot of slot_rows suffix
// rows for its own K/V.  The prefix holds one reference for the parent and one per live child; when
// the count reaches zero the prefix may be freed.  The pool only does the bookkeeping: the K/V rows
// themselves live in caller-owned device buffers, addressed by the rows this pool hands out, and
// fx_branch_pool_batch fills the arrays fx_shared_prefix_decode takes.
#include <stdarg.h>
#include <stdio.h>

#include <mutex>
#include <vector>

#include "fx_internal.h"

namespace {

// record a formatted error message for fx_last_error and return -1
int pool_error(fx_status st, const char* fmt, ...)
{
    char buf[256];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    fx::set_error(st, buf);
    return -1;
}

}  // namespace

struct fx_branch_pool {
    std::mutex mu;
    int prefix_cap = 0, max_branches = 0, slot_rows = 0;
    int prefix_len = 0;
    bool parent_live = true;
    std::vector<int> fork_pos;   // per slot: -1 free, else the child's fork position
    std::vector<int> used;       // per slot: suffix rows written so far
};

extern "C" {

fx_branch_pool* fx_branch_pool_create(int prefix_cap, int max_branches, int slot_rows)
{
    if (prefix_cap < 0 || max_branches < 1 || slot_rows < 0) {
        pool_error(FX_ERR_INVALID_ARG, "need prefix_cap >= 0, max_branches >= 1, slot_rows >= 0");
        return nullptr;
    }
    if ((int64_t)max_branches * slot_rows > 2147483647) {
        pool_error(FX_ERR_INVALID_ARG, "max_branches * slot_rows exceeds the int32 row range");
        return nullptr;
    }
    fx_branch_pool* p = new fx_branch_pool;
    p->prefix_cap = prefix_cap;
    p->max_branches = max_branches;
    p->slot_rows = slot_rows;
    p->fork_pos.assign(max_branches, -1);
    p->used.assign(max_branches, 0);
    return p;
}

void fx_branch_pool_destroy(fx_branch_pool* pool) { delete pool; }

int fx_branch_pool_extend_prefix(fx_branch_pool* pool, int n)
{
    if (!pool || n < 0) return pool_error(FX_ERR_INVALID_ARG, "pool is NULL or n < 0");
    std::lock_guard<std::mutex> lock(pool->mu);
    if (!pool->parent_live) return pool_error(FX_ERR_INVALID_ARG, "the parent branch has been released");
    if (pool->prefix_len + n > pool->prefix_cap)
        return pool_error(FX_ERR_INVALID_ARG, "prefix capacity %d exceeded", pool->prefix_cap);
    const int first = pool->prefix_len;
    pool->prefix_len += n;
    return first;
}

int fx_branch_pool_fork(fx_branch_pool* pool)
{
    if (!pool) return pool_error(FX_ERR_INVALID_ARG, "pool is NULL");
    std::lock_guard<std::mutex> lock(pool->mu);
    if (!pool->parent_live) return pool_error(FX_ERR_INVALID_ARG, "the parent branch has been released");
    for (int s = 0; s < pool->max_branches; ++s) {
        if (pool->fork_pos[s] < 0) {
            pool->fork_pos[s] = pool->prefix_len;
            pool->used[s] = 0;
            return s;
        }
    }
    return pool_error(FX_ERR_UNSUPPORTED, "all %d branch slots are taken", pool->max_branches);
}

int fx_branch_pool_append(fx_branch_pool* pool, int branch, int n)
{
    if (!pool || n < 0) return pool_error(FX_ERR_INVALID_ARG, "pool is NULL or n < 0");
    std::lock_guard<std::mutex> lock(pool->mu);
    if (branch < 0 || branch >= pool->max_branches || pool->fork_pos[branch] < 0)
        return pool_error(FX_ERR_INVALID_ARG, "branch %d is not live", branch);
    if (pool->used[branch] + n > pool->slot_rows)
        return pool_error(FX_ERR_UNSUPPORTED, "branch %d: slot of %d rows is full", branch, pool->slot_rows);
    const int first = branch * pool->slot_rows + pool->used[branch];
    pool->used[branch] += n;
    return first;
}

int fx_branch_pool_release(fx_branch_pool* pool, int branch)
{
    if (!pool) return pool_error(FX_ERR_INVALID_ARG, "pool is NULL");
    std::lock_guard<std::mutex> lock(pool->mu);
    if (branch < 0 || branch >= pool->max_branches || pool->fork_pos[branch] < 0)
        return pool_error(FX_ERR_INVALID_ARG, "branch %d is not live", branch);
    pool->fork_pos[branch] = -1;
    pool->used[branch] = 0;
    int refs = pool->parent_live ? 1 : 0;
    for (int s = 0; s < pool->max_branches; ++s) refs += pool->fork_pos[s] >= 0 ? 1 : 0;
    return refs;
}

int fx_branch_pool_release_parent(fx_branch_pool* pool)
{
    if (!pool) return pool_error(FX_ERR_INVALID_ARG, "pool is NULL");
    std::lock_guard<std::mutex> lock(pool->mu);
    pool->parent_live = false;
    int refs = 0;
    for (int s = 0; s < pool->max_branches; ++s) refs += pool->fork_pos[s] >= 0 ? 1 : 0;
    return refs;
}

int fx_branch_pool_prefix_refs(fx_branch_pool* pool)
{
    if (!pool) return pool_error(FX_ERR_INVALID_ARG, "pool is NULL");
    std::lock_guard<std::mutex> lock(pool->mu);
    int refs = pool->parent_live ? 1 : 0;
    for (int s = 0; s < pool->max_branches; ++s) refs += pool->fork_pos[s] >= 0 ? 1 : 0;
    return refs;
}

int fx_branch_pool_prefix_len(fx_branch_pool* pool)
{
    if (!pool) return pool_error(FX_ERR_INVALID_ARG, "pool is NULL");
    std::lock_guard<std::mutex> lock(pool->mu);
    return pool->prefix_len;
}

int fx_branch_pool_batch(fx_branch_pool* pool, int32_t* ids, int32_t* suf_start, int32_t* suf_len,
                         int32_t* prefix_len)
{
    if (!pool || !ids || !suf_start || !suf_len || !prefix_len)
        return pool_error(FX_ERR_INVALID_ARG, "NULL argument");
    std::lock_guard<std::mutex> lock(pool->mu);
    int n = 0;
    for (int s = 0; s < pool->max_branches; ++s) {
        if (pool->fork_pos[s] < 0) continue;
        ids[n] = s;
        suf_start[n] = s * pool->slot_rows;
        suf_len[n] = pool->used[s];
        prefix_len[n] = pool->fork_pos[s];
        ++n;
    }
    return n;
}

}  // extern "C"
