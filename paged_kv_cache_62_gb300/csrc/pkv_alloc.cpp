// Host-side block allocator for the paged KV cache: which physical blocks
// each sequence's tokens live in, with reference counts for shared blocks.
//
// Semantics (nano-vllm KV-cache post, §3.3 "BlockManager 的设计"):
//  * the free list is a FIFO of block ids, initially 0, 1, ..., num_blocks-1;
//    allocation takes from the front, release appends to the back (§3.3.1);
//  * a block's ref_count is the number of sequences whose table holds it;
//    sharing a block adds one (§3.3.3, the REUSE path);
//  * appending a token that opens a new block (its position is a multiple of
//    block_size) takes a fresh block (§3.3.4, may_append);
//  * writing into a last block that other sequences share first copies it to
//    a fresh block (copy-on-write: §2.2 of the same post; "半满块 COW" in the
//    mini-vLLM README §1); the copy itself is pkv_copy_blocks on the device;
//  * freeing a sequence walks its table backwards, and a block whose count
//    drops to zero goes back to the free list (§3.3.5).
// Prefix hashing (which blocks may be shared) is the caller's decision here:
// sharing is explicit (pkv_allocator_add with a parent, pkv_allocator_fork).
#include <cstdint>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

struct pkv_block_allocator {
    int32_t num_blocks = 0, block_size = 0;
    std::vector<int32_t> ref;    // per block
    std::deque<int32_t> free_q;  // FIFO of free block ids
    struct Seq {
        int32_t tokens = 0;
        std::vector<int32_t> table;
    };
    std::unordered_map<int32_t, Seq> seqs;

    int32_t take()
    {
        const int32_t b = free_q.front();
        free_q.pop_front();
        ref[b] = 1;
        return b;
    }
    void drop(int32_t b)
    {
        if (--ref[b] == 0) free_q.push_back(b);
    }
    int64_t blocks_for(int64_t tokens) const { return (tokens + block_size - 1) / block_size; }
};

namespace {
bool bad(const pkv_block_allocator *a) { return a == nullptr; }
}  // namespace

extern "C" pkv_block_allocator *pkv_allocator_create(int32_t num_blocks, int32_t block_size)
{
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    pkv_block_allocator *a = new (std::nothrow) pkv_block_allocator;
    if (!a) return nullptr;
    try {
        a->num_blocks = num_blocks;
        a->block_size = block_size;
        a->ref.assign(size_t(num_blocks), 0);
        for (int32_t i = 0; i < num_blocks; ++i) a->free_q.push_back(i);
    } catch (...) {
        delete a;
        return nullptr;
    }
    return a;
}

extern "C" void pkv_allocator_destroy(pkv_block_allocator *a) { delete a; }

extern "C" pkv_status pkv_allocator_add(pkv_block_allocator *a, int32_t seq_id, int32_t num_tokens,
                                        int32_t parent_id, int32_t shared_blocks)
{
    if (bad(a) || seq_id < 0 || num_tokens < 0 || shared_blocks < 0) return PKV_EINVAL;
    if (a->seqs.count(seq_id)) return PKV_EINVAL;
    const int64_t need = a->blocks_for(num_tokens);
    const pkv_block_allocator::Seq *parent = nullptr;
    if (shared_blocks > 0) {
        auto it = a->seqs.find(parent_id);
        if (it == a->seqs.end()) return PKV_EINVAL;
        parent = &it->second;
        // only whole blocks the parent holds, and never the block that receives the
        // sequence's last token (that one must be private to be written)
        if (shared_blocks > int64_t(parent->table.size()) || int64_t(shared_blocks) * a->block_size >= num_tokens)
            return PKV_EINVAL;
    }
    if (need - shared_blocks > int64_t(a->free_q.size())) return PKV_EFULL;
    // Everything that may throw happens before any count changes: the table is built (with
    // room for all its blocks) and the entry inserted; moving the table in cannot fail.
    std::vector<int32_t> table;
    try {
        table.reserve(size_t(need));
        if (parent) table.assign(parent->table.begin(), parent->table.begin() + shared_blocks);
        a->seqs.emplace(seq_id, pkv_block_allocator::Seq{});  // may rehash: `parent` is not used below
    } catch (...) {
        return PKV_EFULL;
    }
    pkv_block_allocator::Seq &s = a->seqs.find(seq_id)->second;
    s.tokens = num_tokens;
    s.table = std::move(table);
    for (int32_t b : s.table) ++a->ref[size_t(b)];
    while (int64_t(s.table.size()) < need) s.table.push_back(a->take());
    return PKV_OK;
}

extern "C" pkv_status pkv_allocator_fork(pkv_block_allocator *a, int32_t parent_id, int32_t child_id)
{
    if (bad(a) || child_id < 0 || a->seqs.count(child_id)) return PKV_EINVAL;
    auto it = a->seqs.find(parent_id);
    if (it == a->seqs.end()) return PKV_EINVAL;
    pkv_block_allocator::Seq *c = nullptr;
    try {
        pkv_block_allocator::Seq copy = it->second;
        c = &a->seqs.emplace(child_id, std::move(copy)).first->second;
    } catch (...) {
        a->seqs.erase(child_id);
        return PKV_EFULL;
    }
    for (int32_t b : c->table) ++a->ref[b];
    return PKV_OK;
}

extern "C" pkv_status pkv_allocator_append(pkv_block_allocator *a, int32_t seq_id, int32_t *cow_src,
                                           int32_t *cow_dst)
{
    if (bad(a)) return PKV_EINVAL;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PKV_EINVAL;
    pkv_block_allocator::Seq &s = it->second;
    if (s.tokens == INT32_MAX) return PKV_EINVAL;
    int32_t src = -1, dst = -1;
    const int32_t pos = s.tokens;  // position of the new token
    if (pos % a->block_size == 0) {
        if (a->free_q.empty()) return PKV_EFULL;
        s.table.push_back(a->take());
    } else if (a->ref[s.table.back()] > 1) {
        if (a->free_q.empty()) return PKV_EFULL;
        src = s.table.back();
        dst = a->take();
        --a->ref[src];  // still held by the others: never reaches zero here
        s.table.back() = dst;
    }
    s.tokens = pos + 1;
    if (cow_src) *cow_src = src;
    if (cow_dst) *cow_dst = dst;
    return PKV_OK;
}

extern "C" pkv_status pkv_allocator_free(pkv_block_allocator *a, int32_t seq_id)
{
    if (bad(a)) return PKV_EINVAL;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PKV_EINVAL;
    const std::vector<int32_t> &t = it->second.table;
    for (size_t i = t.size(); i-- > 0;) a->drop(t[i]);
    a->seqs.erase(it);
    return PKV_OK;
}

extern "C" int32_t pkv_allocator_num_free(const pkv_block_allocator *a)
{
    return bad(a) ? -1 : int32_t(a->free_q.size());
}

extern "C" int32_t pkv_allocator_ref_count(const pkv_block_allocator *a, int32_t block_id)
{
    if (bad(a) || block_id < 0 || block_id >= a->num_blocks) return -1;
    return a->ref[size_t(block_id)];
}

extern "C" int32_t pkv_allocator_num_tokens(const pkv_block_allocator *a, int32_t seq_id)
{
    if (bad(a)) return -1;
    auto it = a->seqs.find(seq_id);
    return it == a->seqs.end() ? -1 : it->second.tokens;
}

extern "C" pkv_status pkv_allocator_tables(const pkv_block_allocator *a, const int32_t *seq_ids, int32_t n,
                                           int32_t *block_tables, int32_t max_blocks, int32_t *context_lens)
{
    if (bad(a) || n < 0 || max_blocks <= 0 || (n > 0 && (!seq_ids || !block_tables))) return PKV_EINVAL;
    for (int32_t i = 0; i < n; ++i) {
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end()) return PKV_EINVAL;
        if (int64_t(it->second.table.size()) > max_blocks) return PKV_EBOUNDS;
    }
    for (int32_t i = 0; i < n; ++i) {
        const pkv_block_allocator::Seq &s = a->seqs.find(seq_ids[i])->second;
        int32_t *row = block_tables + int64_t(i) * max_blocks;
        for (int32_t j = 0; j < max_blocks; ++j) row[j] = j < int32_t(s.table.size()) ? s.table[size_t(j)] : -1;
        if (context_lens) context_lens[i] = s.tokens;
    }
    return PKV_OK;
}
