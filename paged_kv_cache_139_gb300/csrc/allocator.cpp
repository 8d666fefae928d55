// Host block allocator: ref-counted physical KV blocks, ceil(len/B)
// allocation on demand, fork / append (with copy-on-write) / free.
//
// "vLLM & PagedAttention: Efficient Memory Management for LLM Serving":
//   §V steps 1-3 (a new physical block only when the last one is full),
//   §VII Figure 8 (reference counts; a write into a shared block copies it
//   first and decrements the old count, the last writer writes in place),
//   §VII Figure 9 (blocks whose count drops to zero are freed),
//   §X (fork, append and free are the sequence primitives).
// "How PagedAttention changed LLM serving throughput": a sequence uses
//   exactly ceil(len / block_size) blocks.
//
// Beam search ("vLLM & PagedAttention" §VII, Figure 9): pkv_beam_step turns
// the current candidates into the next set with fork / append / free (the
// first child of a parent continues its sequence, later children fork it,
// every child appends its token, parents nobody chose are freed last).
//
// Swapping ("vLLM & PagedAttention" §VIII, Figure 4): pkv_move_group moves an
// evicted sequence group to a second allocator (the CPU pool) or back, all or
// nothing, keeping the group's sharing; the caller copies the returned block
// pairs on the device (swap_blocks).
//
// The pages leave open which free block comes next; this allocator hands out
// blocks in a caller-given initial order and re-uses freed blocks last-in,
// first-out (freed in the sequence's logical order).
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "pkv.h"
#include "pkv_internal.h"

struct pkv_allocator {
    int num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> ref;            // reference count per physical block
    std::vector<int32_t> free_stack;     // back() is handed out next
    struct Seq {
        bool live = false;
        int64_t len = 0;
        std::vector<int32_t> blocks;     // logical -> physical
    };
    std::vector<Seq> seqs;               // indexed by sequence id

    int32_t pop() {
        int32_t b = free_stack.back();
        free_stack.pop_back();
        ref[b] = 1;
        return b;
    }
    Seq *get(int32_t id) {
        if (id < 0 || id >= (int32_t)seqs.size() || !seqs[id].live) return nullptr;
        return &seqs[id];
    }
    const Seq *get(int32_t id) const {
        if (id < 0 || id >= (int32_t)seqs.size() || !seqs[id].live) return nullptr;
        return &seqs[id];
    }
};

namespace {

int64_t blocks_needed(int64_t len, int B) { return (len + B - 1) / B; }

// One append; `undo` receives what is needed to revert it.
struct AppendUndo {
    int32_t seq;
    int kind;           // 0 in place, 1 new block pushed, 2 copy-on-write
    int32_t old_block;  // for kind 2
};

pkv_status append_one(pkv_allocator *a, int32_t id, int64_t *slot, int32_t *cow_src,
                      int32_t *cow_dst, AppendUndo *undo) {
    pkv_allocator::Seq *s = a->get(id);
    if (!s) return pkv::fail(PKV_EINVAL, "pkv_seq_append: unknown sequence %d", id);
    const int B = a->block_size;
    const int64_t pos = s->len;
    *cow_src = -1;
    *cow_dst = -1;
    undo->seq = id;
    if (pos % B == 0) {                                 // last block full, or none
        if (a->free_stack.empty())
            return pkv::fail(PKV_ENOMEM, "pkv_seq_append: no free block (sequence %d)", id);
        s->blocks.push_back(a->pop());
        undo->kind = 1;
    } else {
        int32_t last = s->blocks.back();
        if (a->ref[last] > 1) {                         // shared: copy on write
            if (a->free_stack.empty())
                return pkv::fail(PKV_ENOMEM, "pkv_seq_append: no free block for copy-on-write (sequence %d)", id);
            int32_t fresh = a->pop();
            a->ref[last] -= 1;
            s->blocks.back() = fresh;
            *cow_src = last;
            *cow_dst = fresh;
            undo->kind = 2;
            undo->old_block = last;
        } else {
            undo->kind = 0;
        }
    }
    s->len = pos + 1;
    *slot = (int64_t)s->blocks[pos / B] * B + pos % B;
    return PKV_OK;
}

void undo_append(pkv_allocator *a, const AppendUndo &u) {
    pkv_allocator::Seq &s = a->seqs[u.seq];
    s.len -= 1;
    if (u.kind == 1) {
        int32_t b = s.blocks.back();
        s.blocks.pop_back();
        a->ref[b] = 0;
        a->free_stack.push_back(b);
    } else if (u.kind == 2) {
        int32_t fresh = s.blocks.back();
        s.blocks.back() = u.old_block;
        a->ref[u.old_block] += 1;
        a->ref[fresh] = 0;
        a->free_stack.push_back(fresh);
    }
}

}  // namespace

extern "C" {

pkv_status pkv_alloc_create(int num_blocks, int block_size, const int32_t *free_order,
                            pkv_allocator **out) {
    if (!out) return pkv::fail(PKV_EINVAL, "pkv_alloc_create: out is NULL");
    *out = nullptr;
    if (num_blocks < 0 || block_size <= 0)
        return pkv::fail(PKV_EINVAL, "pkv_alloc_create: bad sizes (%d blocks of %d)", num_blocks, block_size);
    pkv_allocator *a = new (std::nothrow) pkv_allocator;
    if (!a) return pkv::fail(PKV_ENOMEM, "pkv_alloc_create: out of host memory");
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->ref.assign(num_blocks, 0);
    a->free_stack.resize(num_blocks);
    if (free_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int i = 0; i < num_blocks; i++) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete a;
                return pkv::fail(PKV_EINVAL, "pkv_alloc_create: free_order is not a permutation (entry %d = %d)", i, b);
            }
            seen[b] = 1;
        }
        for (int i = 0; i < num_blocks; i++) a->free_stack[num_blocks - 1 - i] = free_order[i];
    } else {
        for (int i = 0; i < num_blocks; i++) a->free_stack[num_blocks - 1 - i] = i;
    }
    *out = a;
    return PKV_OK;
}

void pkv_alloc_destroy(pkv_allocator *a) { delete a; }

pkv_status pkv_seq_new(pkv_allocator *a, int64_t len, int32_t *seq) {
    if (!a || !seq || len < 0) return pkv::fail(PKV_EINVAL, "pkv_seq_new: bad argument");
    int64_t n = blocks_needed(len, a->block_size);
    if (n > (int64_t)a->free_stack.size())
        return pkv::fail(PKV_ENOMEM, "pkv_seq_new: need %lld blocks, %zu free", (long long)n, a->free_stack.size());
    pkv_allocator::Seq s;
    s.live = true;
    s.len = len;
    s.blocks.reserve(n);
    for (int64_t i = 0; i < n; i++) s.blocks.push_back(a->pop());
    *seq = (int32_t)a->seqs.size();
    a->seqs.push_back(std::move(s));
    return PKV_OK;
}

pkv_status pkv_seq_fork(pkv_allocator *a, int32_t seq, int32_t *child) {
    if (!a || !child) return pkv::fail(PKV_EINVAL, "pkv_seq_fork: NULL argument");
    const pkv_allocator::Seq *p = a->get(seq);
    if (!p) return pkv::fail(PKV_EINVAL, "pkv_seq_fork: unknown sequence %d", seq);
    pkv_allocator::Seq c;
    c.live = true;
    c.len = p->len;
    c.blocks = p->blocks;
    for (int32_t b : c.blocks) a->ref[b] += 1;
    *child = (int32_t)a->seqs.size();
    a->seqs.push_back(std::move(c));
    return PKV_OK;
}

pkv_status pkv_seq_append(pkv_allocator *a, int32_t seq, int64_t *slot, int32_t *cow_src,
                          int32_t *cow_dst) {
    if (!a || !slot || !cow_src || !cow_dst) return pkv::fail(PKV_EINVAL, "pkv_seq_append: NULL argument");
    AppendUndo u;
    return append_one(a, seq, slot, cow_src, cow_dst, &u);
}

pkv_status pkv_seq_append_batch(pkv_allocator *a, const int32_t *seqs, int n, int64_t *slots,
                                int32_t *cow_pairs, int *num_pairs) {
    if (!a || n < 0 || (n > 0 && (!seqs || !slots || !cow_pairs)) || !num_pairs)
        return pkv::fail(PKV_EINVAL, "pkv_seq_append_batch: bad argument");
    std::vector<AppendUndo> log;
    log.reserve(n);
    int np = 0;
    for (int i = 0; i < n; i++) {
        int32_t src, dst;
        AppendUndo u;
        pkv_status st = append_one(a, seqs[i], &slots[i], &src, &dst, &u);
        if (st != PKV_OK) {
            for (int j = (int)log.size() - 1; j >= 0; j--) undo_append(a, log[j]);
            return st;
        }
        log.push_back(u);
        if (src >= 0) {
            cow_pairs[2 * np] = src;
            cow_pairs[2 * np + 1] = dst;
            np++;
        }
    }
    *num_pairs = np;
    return PKV_OK;
}

pkv_status pkv_seq_free(pkv_allocator *a, int32_t seq) {
    if (!a) return pkv::fail(PKV_EINVAL, "pkv_seq_free: NULL allocator");
    pkv_allocator::Seq *s = a->get(seq);
    if (!s) return pkv::fail(PKV_EINVAL, "pkv_seq_free: unknown sequence %d", seq);
    for (int32_t b : s->blocks) {
        if (--a->ref[b] == 0) a->free_stack.push_back(b);
    }
    s->live = false;
    s->blocks.clear();
    s->blocks.shrink_to_fit();
    s->len = 0;
    return PKV_OK;
}

pkv_status pkv_seq_len(const pkv_allocator *a, int32_t seq, int64_t *len) {
    if (!a || !len) return pkv::fail(PKV_EINVAL, "pkv_seq_len: NULL argument");
    const pkv_allocator::Seq *s = a->get(seq);
    if (!s) return pkv::fail(PKV_EINVAL, "pkv_seq_len: unknown sequence %d", seq);
    *len = s->len;
    return PKV_OK;
}

pkv_status pkv_seq_block_table(const pkv_allocator *a, int32_t seq, int32_t *out, int cap, int *n) {
    if (!a || !n || cap < 0 || (cap > 0 && !out)) return pkv::fail(PKV_EINVAL, "pkv_seq_block_table: bad argument");
    const pkv_allocator::Seq *s = a->get(seq);
    if (!s) return pkv::fail(PKV_EINVAL, "pkv_seq_block_table: unknown sequence %d", seq);
    int m = (int)s->blocks.size();
    *n = m;
    if (m > cap) return pkv::fail(PKV_EINVAL, "pkv_seq_block_table: table of %d entries, room for %d", m, cap);
    if (m) std::memcpy(out, s->blocks.data(), sizeof(int32_t) * m);
    return PKV_OK;
}

pkv_status pkv_build_block_tables(const pkv_allocator *a, const int32_t *seqs, int n,
                                  int32_t *tables, int max_blocks, int32_t *context_lens) {
    if (!a || n < 0 || max_blocks < 0 || (n > 0 && (!seqs || !context_lens || (max_blocks > 0 && !tables))))
        return pkv::fail(PKV_EINVAL, "pkv_build_block_tables: bad argument");
    for (int i = 0; i < n; i++) {
        const pkv_allocator::Seq *s = a->get(seqs[i]);
        if (!s) return pkv::fail(PKV_EINVAL, "pkv_build_block_tables: unknown sequence %d", seqs[i]);
        int m = (int)s->blocks.size();
        if (m > max_blocks || s->len > INT32_MAX)
            return pkv::fail(PKV_EINVAL, "pkv_build_block_tables: sequence %d has %d blocks, table width %d", seqs[i], m, max_blocks);
        int32_t *row = tables + (int64_t)i * max_blocks;
        for (int j = 0; j < m; j++) row[j] = s->blocks[j];
        for (int j = m; j < max_blocks; j++) row[j] = -1;
        context_lens[i] = (int32_t)s->len;
    }
    return PKV_OK;
}

pkv_status pkv_beam_step(pkv_allocator *a, const int32_t *beams, int k, const int32_t *parents, int kn,
                         int32_t *new_beams, int64_t *slots, int32_t *cow_pairs, int *num_pairs) {
    if (!a || k < 0 || kn < 0 || (k > 0 && !beams) || (kn > 0 && (!parents || !new_beams || !slots || !cow_pairs)) ||
        !num_pairs)
        return pkv::fail(PKV_EINVAL, "pkv_beam_step: bad argument");
    *num_pairs = 0;
    std::vector<char> seen(a->seqs.size(), 0);
    for (int i = 0; i < k; i++) {
        if (!a->get(beams[i]) || seen[beams[i]])
            return pkv::fail(PKV_EINVAL, "pkv_beam_step: unknown or repeated beam %d", beams[i]);
        seen[beams[i]] = 1;
    }
    for (int i = 0; i < kn; i++)
        if (parents[i] < 0 || parents[i] >= k)
            return pkv::fail(PKV_EINVAL, "pkv_beam_step: parent index %d of candidate %d out of range", parents[i], i);
    const size_t nseq0 = a->seqs.size();
    std::vector<char> taken(k, 0);
    for (int i = 0; i < kn; i++) {
        const int p = parents[i];
        if (!taken[p]) {
            taken[p] = 1;
            new_beams[i] = beams[p];
        } else {
            pkv_status st = pkv_seq_fork(a, beams[p], &new_beams[i]);
            if (st != PKV_OK) return st;           // cannot happen: the parent is live
        }
    }
    std::vector<AppendUndo> log;
    log.reserve(kn);
    int np = 0;
    for (int i = 0; i < kn; i++) {
        int32_t src, dst;
        AppendUndo u;
        pkv_status st = append_one(a, new_beams[i], &slots[i], &src, &dst, &u);
        if (st != PKV_OK) {
            // undo the appends, then the forks (children take the newest ids)
            for (int j = (int)log.size() - 1; j >= 0; j--) undo_append(a, log[j]);
            while (a->seqs.size() > nseq0) {
                for (int32_t b : a->seqs.back().blocks) a->ref[b] -= 1;
                a->seqs.pop_back();
            }
            return st;
        }
        log.push_back(u);
        if (src >= 0) {
            cow_pairs[2 * np] = src;
            cow_pairs[2 * np + 1] = dst;
            np++;
        }
    }
    for (int i = 0; i < k; i++)
        if (!taken[i]) pkv_seq_free(a, beams[i]);
    *num_pairs = np;
    return PKV_OK;
}

int pkv_blocks_in_use(const pkv_allocator *a) { return a ? a->num_blocks - (int)a->free_stack.size() : -1; }

pkv_status pkv_move_group(pkv_allocator *src, pkv_allocator *dst, const int32_t *seqs, int n, int32_t *new_ids,
                          int32_t *pairs, int pairs_cap, int *num_pairs) {
    if (!src || !dst || src == dst || n < 0 || (n > 0 && (!seqs || !new_ids)) || !num_pairs || pairs_cap < 0 ||
        (pairs_cap > 0 && !pairs))
        return pkv::fail(PKV_EINVAL, "pkv_move_group: bad argument");
    *num_pairs = 0;
    if (src->block_size != dst->block_size)
        return pkv::fail(PKV_EINVAL, "pkv_move_group: block sizes differ (%d and %d)", src->block_size,
                         dst->block_size);
    // distinct blocks in first-seen order, and how often the group uses each
    std::vector<int32_t> uses(src->num_blocks, 0), order;
    std::vector<char> seen_seq(src->seqs.size(), 0);
    for (int i = 0; i < n; i++) {
        const pkv_allocator::Seq *s = src->get(seqs[i]);
        if (!s || seen_seq[seqs[i]]) return pkv::fail(PKV_EINVAL, "pkv_move_group: unknown or repeated sequence %d", seqs[i]);
        seen_seq[seqs[i]] = 1;
        for (int32_t b : s->blocks) {
            if (uses[b]++ == 0) order.push_back(b);
        }
    }
    for (int32_t b : order)
        if (src->ref[b] != uses[b])
            return pkv::fail(PKV_EINVAL, "pkv_move_group: block %d is shared with a sequence outside the group", b);
    if (order.size() > dst->free_stack.size())
        return pkv::fail(PKV_ENOMEM, "pkv_move_group: need %zu blocks in the other pool, %zu free", order.size(),
                         dst->free_stack.size());
    if ((int64_t)order.size() > pairs_cap)
        return pkv::fail(PKV_EINVAL, "pkv_move_group: %zu pairs, room for %d", order.size(), pairs_cap);
    std::vector<int32_t> remap(src->num_blocks, -1);
    for (size_t k = 0; k < order.size(); k++) {
        const int32_t b = order[k];
        const int32_t c = dst->pop();
        dst->ref[c] = uses[b];
        remap[b] = c;
        pairs[2 * k] = b;
        pairs[2 * k + 1] = c;
    }
    for (int i = 0; i < n; i++) {
        const pkv_allocator::Seq &s = src->seqs[seqs[i]];
        pkv_allocator::Seq m;
        m.live = true;
        m.len = s.len;
        m.blocks.reserve(s.blocks.size());
        for (int32_t b : s.blocks) m.blocks.push_back(remap[b]);
        new_ids[i] = (int32_t)dst->seqs.size();
        dst->seqs.push_back(std::move(m));
    }
    for (int i = 0; i < n; i++) pkv_seq_free(src, seqs[i]);
    *num_pairs = (int)order.size();
    return PKV_OK;
}

int pkv_block_ref(const pkv_allocator *a, int32_t block) {
    if (!a || block < 0 || block >= a->num_blocks) return -1;
    return a->ref[block];
}

int pkv_num_free(const pkv_allocator *a) { return a ? (int)a->free_stack.size() : -1; }

pkv_status pkv_free_list(const pkv_allocator *a, int32_t *out, int cap, int *n) {
    if (!a || !n || cap < 0 || (cap > 0 && !out)) return pkv::fail(PKV_EINVAL, "pkv_free_list: bad argument");
    int m = (int)a->free_stack.size();
    *n = m;
    int k = m < cap ? m : cap;
    for (int i = 0; i < k; i++) out[i] = a->free_stack[m - 1 - i];
    return PKV_OK;
}

}  // extern "C"
