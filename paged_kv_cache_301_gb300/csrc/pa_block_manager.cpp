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
#include <stdint.h>

#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedattn.h"

struct pa_block_manager {
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> stack;      // free ids, top = back()
  std::vector<int32_t> refs;       // refcount per id, 0 = free
  struct Seq {
    std::vector<int32_t> table;
    int len = 0;
    bool live = false;
  };
  std::vector<Seq> seqs;

  int blocks_for(int tokens) const { return (tokens + block_size - 1) / block_size; }

  pa_status take(int n, int32_t* out) {
    if (n < 0) return PA_ERR_INVALID_ARG;
    if ((size_t)n > stack.size()) return PA_ERR_OUT_OF_BLOCKS;
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
    for (int i = 0; i < n; ++i) {
      if (--refs[ids[i]] == 0) stack.push_back(ids[i]);
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
