// Host-side refcounted block manager of libpagedattn.
//
// Rules ("10 — Paged Attention" tutorial, §4 "Tiny example"; copy-on-write from
// §5 "Copy-on-write sharing" and the subroutine-cs article §3):
//   * free ids form a LIFO stack; by default ids num_blocks-1 .. 0 are pushed in
//     that order, so id 0 is handed out first;
//   * an allocation of n takes the n topmost ids, in the order they sit in the
//     stack, and sets their refcount to 1; a shortage fails with no change;
//   * a free drops each refcount and pushes the id back when it reaches 0;
//   * a fork raises the refcount of every id of a table;
//   * a sequence of length L owns ceil(L / block_size) blocks; appending a token
//     either opens one new block (at a block boundary) or, when the token's
//     block is shared, clones it first (copy-on-write).
// Every operation validates before it mutates, so a failed call leaves the
// manager unchanged.
//
// Prefix cache (tutorial §5 "The relationship to prefix caching"): full blocks
// of a prompt are keyed by a hash of the whole prefix up to and including the
// block, key_i = FNV-1a-64(key_{i-1} as 8 little-endian bytes, then the block's
// token ids as 4 little-endian bytes each), key_{-1} = 0.  A new prompt points
// its leading blocks at cached blocks with the same keys (and the same parent
// key and token ids) and raises their refcounts, up to the first miss; its other
// full blocks are registered.  A cached block whose refcount reaches zero waits
// on an eviction queue, where it can still be hit; blocks reaching zero in one
// release join the queue last block first.  An allocation that finds the free
// stack short evicts from the front of the queue onto the stack first.
#include <stdint.h>

#include <iterator>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedattn.h"

struct pa_block_manager {
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> stack;      // free ids, top = back()
  std::vector<int32_t> refs;       // refcount per id, 0 = free or queued for eviction
  struct Seq {
    std::vector<int32_t> table;
    int len = 0;
    bool live = false;
  };
  std::vector<Seq> seqs;

  // prefix cache
  struct Entry {
    uint64_t key = 0, parent = 0;
    std::vector<int32_t> tokens;
    bool cached = false;
  };
  std::vector<Entry> entry;                                   // per block id
  std::unordered_map<uint64_t, int32_t> block_of;             // key -> block id
  std::list<int32_t> queue;                                   // refcount-0 cached blocks
  std::vector<std::list<int32_t>::iterator> qpos;             // position while queued
  std::vector<char> queued;

  int blocks_for(int tokens) const { return (tokens + block_size - 1) / block_size; }

  void evict_front() {
    const int32_t id = queue.front();
    queue.pop_front();
    queued[id] = 0;
    block_of.erase(entry[id].key);
    entry[id] = Entry();
    stack.push_back(id);
  }

  pa_status take(int n, int32_t* out) {
    if (n < 0) return PA_ERR_INVALID_ARG;
    if ((size_t)n > stack.size() + queue.size()) return PA_ERR_OUT_OF_BLOCKS;
    while (stack.size() < (size_t)n) evict_front();
    const size_t first = stack.size() - (size_t)n;
    for (int i = 0; i < n; ++i) {
      const int32_t id = stack[first + i];
      out[i] = id;
      refs[id] = 1;
    }
    stack.resize(first);
    return PA_OK;
  }

  bool in_range(int32_t id) const { return id >= 0 && id < num_blocks; }

  pa_status release(const int32_t* ids, int n) {
    // validate first: an id listed k times needs refcount >= k
    std::unordered_map<int32_t, int> uses;
    for (int i = 0; i < n; ++i) {
      if (!in_range(ids[i])) return PA_ERR_BLOCK_STATE;
      if (++uses[ids[i]] > refs[ids[i]]) return PA_ERR_BLOCK_STATE;
    }
    std::vector<int32_t> parked;
    for (int i = 0; i < n; ++i) {
      if (--refs[ids[i]] == 0) {
        if (entry[ids[i]].cached) parked.push_back(ids[i]);
        else stack.push_back(ids[i]);
      }
    }
    for (auto it = parked.rbegin(); it != parked.rend(); ++it) {
      queue.push_back(*it);
      qpos[*it] = std::prev(queue.end());
      queued[*it] = 1;
    }
    return PA_OK;
  }

  pa_status share(const int32_t* ids, int n) {
    for (int i = 0; i < n; ++i)
      if (!in_range(ids[i]) || refs[ids[i]] <= 0) return PA_ERR_BLOCK_STATE;
    for (int i = 0; i < n; ++i) ++refs[ids[i]];
    return PA_OK;
  }

  Seq* seq(int id) {
    if (id < 0 || (size_t)id >= seqs.size() || !seqs[id].live) return nullptr;
    return &seqs[id];
  }
};

extern "C" pa_status pa_bm_create(int num_blocks, int block_size,
                                  const int32_t* initial_free_stack, pa_block_manager** out) {
  if (!out || num_blocks < 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
  *out = nullptr;
  pa_block_manager* bm = new (std::nothrow) pa_block_manager();
  if (!bm) return PA_ERR_INVALID_ARG;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->refs.assign((size_t)num_blocks, 0);
  bm->entry.resize((size_t)num_blocks);
  bm->qpos.resize((size_t)num_blocks);
  bm->queued.assign((size_t)num_blocks, 0);
  bm->stack.resize((size_t)num_blocks);
  if (initial_free_stack) {
    std::vector<char> seen((size_t)num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) {
      const int32_t id = initial_free_stack[i];
      if (id < 0 || id >= num_blocks || seen[id]) {
        delete bm;
        return PA_ERR_INVALID_ARG;
      }
      seen[id] = 1;
      bm->stack[i] = id;
    }
  } else {
    for (int i = 0; i < num_blocks; ++i) bm->stack[i] = num_blocks - 1 - i;
  }
  *out = bm;
  return PA_OK;
}

extern "C" void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

extern "C" int pa_bm_num_free(const pa_block_manager* bm) {
  return bm ? (int)bm->stack.size() : -1;
}

extern "C" int pa_bm_num_evictable(const pa_block_manager* bm) {
  return bm ? (int)bm->queue.size() : -1;
}

extern "C" int pa_bm_refcount(const pa_block_manager* bm, int block_id) {
  if (!bm || !bm->in_range(block_id)) return -1;
  return bm->refs[block_id];
}

extern "C" pa_status pa_bm_allocate(pa_block_manager* bm, int n, int32_t* out_ids) {
  if (!bm || (n > 0 && !out_ids)) return PA_ERR_INVALID_ARG;
  return bm->take(n, out_ids);
}

extern "C" pa_status pa_bm_free(pa_block_manager* bm, const int32_t* ids, int n) {
  if (!bm || n < 0 || (n > 0 && !ids)) return PA_ERR_INVALID_ARG;
  return bm->release(ids, n);
}

extern "C" pa_status pa_bm_fork(pa_block_manager* bm, const int32_t* ids, int n) {
  if (!bm || n < 0 || (n > 0 && !ids)) return PA_ERR_INVALID_ARG;
  return bm->share(ids, n);
}

extern "C" pa_status pa_bm_seq_create(pa_block_manager* bm, int prompt_len, int* seq_id) {
  if (!bm || !seq_id || prompt_len < 0) return PA_ERR_INVALID_ARG;
  pa_block_manager::Seq s;
  s.table.resize((size_t)bm->blocks_for(prompt_len));
  const pa_status st = bm->take((int)s.table.size(), s.table.data());
  if (st != PA_OK) return st;
  s.len = prompt_len;
  s.live = true;
  bm->seqs.push_back(std::move(s));
  *seq_id = (int)bm->seqs.size() - 1;
  return PA_OK;
}

extern "C" pa_status pa_bm_seq_fork(pa_block_manager* bm, int parent, int* child) {
  if (!bm || !child) return PA_ERR_INVALID_ARG;
  pa_block_manager::Seq* p = bm->seq(parent);
  if (!p) return PA_ERR_BLOCK_STATE;
  pa_block_manager::Seq c;
  c.table = p->table;
  c.len = p->len;
  c.live = true;
  const pa_status st = bm->share(c.table.data(), (int)c.table.size());
  if (st != PA_OK) return st;
  bm->seqs.push_back(std::move(c));
  *child = (int)bm->seqs.size() - 1;
  return PA_OK;
}

extern "C" pa_status pa_bm_seq_release(pa_block_manager* bm, int seq_id) {
  if (!bm) return PA_ERR_INVALID_ARG;
  pa_block_manager::Seq* s = bm->seq(seq_id);
  if (!s) return PA_ERR_BLOCK_STATE;
  const pa_status st = bm->release(s->table.data(), (int)s->table.size());
  if (st != PA_OK) return st;
  s->table.clear();
  s->len = 0;
  s->live = false;
  return PA_OK;
}

extern "C" pa_status pa_bm_seq_append(pa_block_manager* bm, int seq_id, int32_t* slot,
                                      int32_t* cow_src, int32_t* cow_dst) {
  if (!bm || !slot || !cow_src || !cow_dst) return PA_ERR_INVALID_ARG;
  pa_block_manager::Seq* s = bm->seq(seq_id);
  if (!s) return PA_ERR_BLOCK_STATE;
  const int pos = s->len;
  const int idx = pos / bm->block_size;
  int32_t src = -1, dst = -1;
  if (idx == (int)s->table.size()) {            // crossing into a new block
    int32_t fresh;
    const pa_status st = bm->take(1, &fresh);
    if (st != PA_OK) return st;
    s->table.push_back(fresh);
  } else if (bm->refs[s->table[idx]] > 1) {     // shared block: clone before writing
    int32_t fresh;
    const pa_status st = bm->take(1, &fresh);
    if (st != PA_OK) return st;
    src = s->table[idx];
    dst = fresh;
    --bm->refs[src];                            // stays >= 1: still referenced
    s->table[idx] = fresh;
  }
  s->len = pos + 1;
  *slot = s->table[idx] * bm->block_size + pos % bm->block_size;
  *cow_src = src;
  *cow_dst = dst;
  return PA_OK;
}

extern "C" int pa_bm_seq_len(const pa_block_manager* bm, int seq_id) {
  if (!bm || seq_id < 0 || (size_t)seq_id >= bm->seqs.size() || !bm->seqs[seq_id].live)
    return -1;
  return bm->seqs[seq_id].len;
}

extern "C" int pa_bm_seq_num_blocks(const pa_block_manager* bm, int seq_id) {
  if (!bm || seq_id < 0 || (size_t)seq_id >= bm->seqs.size() || !bm->seqs[seq_id].live)
    return -1;
  return (int)bm->seqs[seq_id].table.size();
}

extern "C" pa_status pa_bm_export(const pa_block_manager* bm, const int* seq_ids, int n,
                                  int max_blocks, int32_t pad_id, int32_t* block_tables,
                                  int32_t* seq_lens) {
  if (!bm || n < 0 || max_blocks <= 0 || (n > 0 && (!seq_ids || !block_tables || !seq_lens)))
    return PA_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const int id = seq_ids[i];
    if (id < 0 || (size_t)id >= bm->seqs.size() || !bm->seqs[id].live) return PA_ERR_BLOCK_STATE;
    if ((int)bm->seqs[id].table.size() > max_blocks) return PA_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n; ++i) {
    const pa_block_manager::Seq& s = bm->seqs[seq_ids[i]];
    int32_t* row = block_tables + (int64_t)i * max_blocks;
    for (int j = 0; j < max_blocks; ++j)
      row[j] = j < (int)s.table.size() ? s.table[j] : pad_id;
    seq_lens[i] = s.len;
  }
  return PA_OK;
}

namespace {

constexpr uint64_t kFnvOffset = 0xCBF29CE484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001B3ull;

// FNV-1a over the low `nbytes` bytes of v, least significant byte first.
uint64_t fnv1a_le(uint64_t h, uint64_t v, int nbytes) {
  for (int i = 0; i < nbytes; ++i) {
    h ^= (v >> (8 * i)) & 0xFFu;
    h *= kFnvPrime;
  }
  return h;
}

uint64_t block_key(uint64_t parent, const int32_t* tokens, int n) {
  uint64_t h = fnv1a_le(kFnvOffset, parent, 8);
  for (int i = 0; i < n; ++i) h = fnv1a_le(h, (uint64_t)(uint32_t)tokens[i], 4);
  return h;
}

}  // namespace

extern "C" pa_status pa_bm_seq_create_cached(pa_block_manager* bm, const int32_t* token_ids,
                                             int num_tokens, int* seq_id, int* cached_tokens) {
  if (!bm || !seq_id || !cached_tokens || num_tokens < 0 || (num_tokens > 0 && !token_ids))
    return PA_ERR_INVALID_ARG;
  const int bs = bm->block_size;
  const int full = num_tokens / bs;
  std::vector<uint64_t> keys((size_t)full), parents((size_t)full);
  uint64_t parent = 0;
  for (int i = 0; i < full; ++i) {
    parents[i] = parent;
    keys[i] = block_key(parent, token_ids + (int64_t)i * bs, bs);
    parent = keys[i];
  }
  std::vector<int32_t> table;
  for (int i = 0; i < full; ++i) {
    auto it = bm->block_of.find(keys[i]);
    if (it == bm->block_of.end()) break;
    const pa_block_manager::Entry& e = bm->entry[it->second];
    bool same = e.parent == parents[i];
    for (int j = 0; same && j < bs; ++j) same = e.tokens[j] == token_ids[(int64_t)i * bs + j];
    if (!same) break;
    table.push_back(it->second);
  }
  const int hits = (int)table.size();
  const int need = bm->blocks_for(num_tokens) - hits;
  size_t queued_hits = 0;
  for (int32_t b : table) queued_hits += bm->refs[b] == 0;
  if ((size_t)need > bm->stack.size() + bm->queue.size() - queued_hits)
    return PA_ERR_OUT_OF_BLOCKS;
  for (int32_t b : table) {
    if (bm->refs[b] > 0) {
      ++bm->refs[b];
    } else {
      bm->queue.erase(bm->qpos[b]);
      bm->queued[b] = 0;
      bm->refs[b] = 1;
    }
  }
  table.resize((size_t)(hits + need));
  const pa_status st = bm->take(need, table.data() + hits);   // cannot fail: checked above
  if (st != PA_OK) return st;
  for (int i = hits; i < full; ++i) {
    if (bm->block_of.count(keys[i])) continue;
    const int32_t b = table[i];
    bm->block_of[keys[i]] = b;
    pa_block_manager::Entry& e = bm->entry[b];
    e.key = keys[i];
    e.parent = parents[i];
    e.tokens.assign(token_ids + (int64_t)i * bs, token_ids + (int64_t)(i + 1) * bs);
    e.cached = true;
  }
  pa_block_manager::Seq s;
  s.table = std::move(table);
  s.len = num_tokens;
  s.live = true;
  bm->seqs.push_back(std::move(s));
  *seq_id = (int)bm->seqs.size() - 1;
  *cached_tokens = hits * bs;
  return PA_OK;
}
