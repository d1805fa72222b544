// Host runtime: paged-KV block allocator and continuous-batching scheduler (cb_sched.h).
//
// Block allocator ("LLM learning path 3.3 Batching & Memory Management", sections "Code" and
// "PagedAttention: block tables"): a stack of free blocks, a reference count per block, block
// tables per sequence; growing a sequence takes a new block when its last block is full and
// copies the last block first when it is shared (copy-on-write); fork shares every block.
//
// Scheduler (transformers "Continuous batching architecture", section "Scheduler" and its
// chunked-prefill paragraph): every step admits work in policy order under a token budget,
// a request cap and the free blocks; a prompt that does not fit the remaining token budget is
// processed as far as it fits and continued on later steps.
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <new>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "cb_sched.h"

namespace cb {
cb_status set_last_error(cb_status st, const char* msg);
}  // namespace cb

namespace {

cb_status fail(cb_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
cb_status fail(cb_status st, const char* fmt, ...) {
  char buf[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  return cb::set_last_error(st, buf);
}

struct SeqBlocks {
  std::vector<int32_t> blocks;
  int32_t len = 0;     // tokens held
  int32_t hashed = 0;  // leading blocks whose content hash chain is known
  uint64_t chain = 0;  // hash of block hashed - 1 (0 before the first)
};

// Content hash of one full block chained with the hash of everything before it: 64-bit
// FNV-1a over the parent hash's 8 bytes, then each token id's 4 bytes, little-endian.
uint64_t block_hash(uint64_t parent, const int32_t* tokens, int32_t n) {
  uint64_t h = 14695981039346656037ull;
  auto mix = [&](uint64_t x, int bytes) {
    for (int i = 0; i < bytes; ++i) {
      h ^= (x >> (8 * i)) & 0xffu;
      h *= 1099511628211ull;
    }
  };
  mix(parent, 8);
  for (int32_t i = 0; i < n; ++i) mix((uint32_t)tokens[i], 4);
  return h;
}

}  // namespace

struct cb_alloc {
  int32_t num_blocks = 0, bs = 0, max_blocks = 0;
  std::vector<int32_t> free_stack;  // blocks without cached content; top = back
  std::vector<int32_t> ref;
  std::unordered_map<int32_t, SeqBlocks> seqs;
  // Prefix cache ("Continuous batching architecture", sections "Prefix caching" and
  // "Eviction"): every completed prompt block gets a content hash; a free block keeps its
  // content and hash ("initialized") until an allocation finds no block without content, and
  // then the most recently initialized free block is demoted (its hash dropped) and reused.
  bool prefix = false;
  std::vector<uint64_t> bhash;                    // 0: no cached content
  std::vector<uint64_t> bparent;                  // chain hash before the block
  std::vector<std::vector<int32_t>> btokens;      // the block's token ids
  std::vector<int64_t> stamp;                     // order of initialization
  std::unordered_map<uint64_t, int32_t> by_hash;  // content hash -> block
  std::set<std::pair<int64_t, int32_t>> init_free;  // (stamp, block), free and initialized
  int64_t next_stamp = 1;

  int32_t free_count() const { return (int32_t)(free_stack.size() + init_free.size()); }
  void drop_hash(int32_t b) {
    auto it = by_hash.find(bhash[b]);
    if (it != by_hash.end() && it->second == b) by_hash.erase(it);
    bhash[b] = 0;
  }
  int32_t pop() {
    int32_t b;
    if (!free_stack.empty()) {
      b = free_stack.back();
      free_stack.pop_back();
    } else {
      auto last = std::prev(init_free.end());  // the most recently initialized free block
      b = last->second;
      init_free.erase(last);
      drop_hash(b);
    }
    ref[b] = 1;
    return b;
  }
  void release(int32_t b) {  // reference count reached 0
    if (prefix && bhash[b] != 0) init_free.insert({stamp[b], b});
    else free_stack.push_back(b);
  }
  void retain(int32_t b) {  // a cached block is taken by one more sequence
    if (ref[b] == 0) init_free.erase({stamp[b], b});
    ref[b] += 1;
  }
  static int32_t blocks_for(int64_t tokens, int32_t bs) { return (int32_t)((tokens + bs - 1) / bs); }
  // Blocks growing `sq` by n tokens takes: new blocks past the last one, plus one copy when
  // the first token lands in a partly filled, shared last block.
  int32_t needed(const SeqBlocks& sq, int32_t n) const {
    if (n <= 0) return 0;
    const int32_t grow = blocks_for((int64_t)sq.len + n, bs) - (int32_t)sq.blocks.size();
    const bool cow = (sq.len % bs) != 0 && ref[sq.blocks.back()] > 1;
    return grow + (cow ? 1 : 0);
  }
};

struct cb_sched {
  enum State { kWaiting, kPrefill, kDecode, kDone };
  struct Request {
    int32_t id, prompt, max_new;
    int32_t done = 0;       // prompt tokens already in the cache
    int32_t generated = 0;  // tokens produced so far
    State state = kWaiting;
    std::vector<int32_t> tokens;  // prompt token ids (prefix caching), may be empty
  };
  cb_alloc* alloc = nullptr;
  cb_sched_config cfg{};
  std::vector<Request> reqs;  // arrival order (forks appended when created)
  std::unordered_map<int32_t, size_t> index;
};

extern "C" {

// ------------------------------------------------------------------------------- allocator

cb_status cb_alloc_create(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                          cb_alloc** out) {
  if (out == nullptr) return fail(CB_ERR_INVALID_ARG, "cb_alloc_create: out is NULL");
  *out = nullptr;
  if (num_blocks < 1 || block_size < 4 || max_blocks_per_seq < 1)
    return fail(CB_ERR_INVALID_ARG,
                "cb_alloc_create: need num_blocks >= 1, block_size >= 4, max_blocks_per_seq >= 1");
  cb_alloc* a = new (std::nothrow) cb_alloc;
  if (a == nullptr) return fail(CB_ERR_INVALID_ARG, "cb_alloc_create: out of host memory");
  a->num_blocks = num_blocks;
  a->bs = block_size;
  a->max_blocks = max_blocks_per_seq;
  a->free_stack.resize(num_blocks);
  for (int32_t i = 0; i < num_blocks; ++i) a->free_stack[i] = i;  // block num_blocks-1 on top
  a->ref.assign(num_blocks, 0);
  a->bhash.assign(num_blocks, 0);
  a->bparent.assign(num_blocks, 0);
  a->btokens.resize(num_blocks);
  a->stamp.assign(num_blocks, 0);
  *out = a;
  return CB_OK;
}

void cb_alloc_destroy(cb_alloc* a) { delete a; }

cb_status cb_alloc_add_seq(cb_alloc* a, int32_t seq, int32_t n_tokens) {
  if (a == nullptr || n_tokens < 0) return fail(CB_ERR_INVALID_ARG, "cb_alloc_add_seq: bad argument");
  if (a->seqs.count(seq)) return fail(CB_ERR_INVALID_ARG, "cb_alloc_add_seq: sequence %d exists", seq);
  const int32_t nb = cb_alloc::blocks_for(n_tokens, a->bs);
  if (nb > a->max_blocks)
    return fail(CB_ERR_OUT_OF_RANGE, "cb_alloc_add_seq: %d blocks exceed max_blocks_per_seq %d", nb,
                a->max_blocks);
  if (nb > a->free_count())
    return fail(CB_ERR_OUT_OF_RANGE, "cb_alloc_add_seq: %d blocks needed, %d free", nb,
                a->free_count());
  SeqBlocks sq;
  sq.len = n_tokens;
  sq.blocks.reserve(nb);
  for (int32_t i = 0; i < nb; ++i) sq.blocks.push_back(a->pop());
  a->seqs.emplace(seq, std::move(sq));
  return CB_OK;
}

int32_t cb_alloc_blocks_needed(const cb_alloc* a, int32_t seq, int32_t n_tokens) {
  if (a == nullptr || n_tokens <= 0) return 0;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return cb_alloc::blocks_for(n_tokens, a->bs);
  return a->needed(it->second, n_tokens);
}

cb_status cb_alloc_append(cb_alloc* a, int32_t seq, int32_t n_tokens, int32_t* cow_src,
                          int32_t* cow_dst, int32_t* n_cow) {
  if (n_cow != nullptr) *n_cow = 0;
  if (a == nullptr || n_tokens < 0) return fail(CB_ERR_INVALID_ARG, "cb_alloc_append: bad argument");
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return fail(CB_ERR_INVALID_ARG, "cb_alloc_append: no sequence %d", seq);
  SeqBlocks& sq = it->second;
  if (n_tokens == 0) return CB_OK;
  const int32_t total = cb_alloc::blocks_for((int64_t)sq.len + n_tokens, a->bs);
  if (total > a->max_blocks)
    return fail(CB_ERR_OUT_OF_RANGE, "cb_alloc_append: %d blocks exceed max_blocks_per_seq %d",
                total, a->max_blocks);
  const int32_t need = a->needed(sq, n_tokens);
  if (need > a->free_count())
    return fail(CB_ERR_OUT_OF_RANGE, "cb_alloc_append: %d blocks needed, %d free", need,
                a->free_count());
  if (sq.len % a->bs != 0 && a->ref[sq.blocks.back()] > 1) {
    if (cow_src == nullptr || cow_dst == nullptr)
      return fail(CB_ERR_INVALID_ARG, "cb_alloc_append: a copy-on-write is needed but no output");
    const int32_t old = sq.blocks.back();
    a->ref[old] -= 1;
    const int32_t fresh = a->pop();
    sq.blocks.back() = fresh;
    cow_src[0] = old;
    cow_dst[0] = fresh;
    if (n_cow != nullptr) *n_cow = 1;
  }
  while ((int32_t)sq.blocks.size() < total) sq.blocks.push_back(a->pop());
  sq.len += n_tokens;
  return CB_OK;
}

cb_status cb_alloc_fork(cb_alloc* a, int32_t parent, int32_t child) {
  if (a == nullptr) return fail(CB_ERR_INVALID_ARG, "cb_alloc_fork: NULL allocator");
  auto it = a->seqs.find(parent);
  if (it == a->seqs.end()) return fail(CB_ERR_INVALID_ARG, "cb_alloc_fork: no sequence %d", parent);
  if (a->seqs.count(child)) return fail(CB_ERR_INVALID_ARG, "cb_alloc_fork: sequence %d exists", child);
  SeqBlocks sq = it->second;
  for (int32_t b : sq.blocks) a->ref[b] += 1;
  a->seqs.emplace(child, std::move(sq));
  return CB_OK;
}

cb_status cb_alloc_free_seq(cb_alloc* a, int32_t seq) {
  if (a == nullptr) return fail(CB_ERR_INVALID_ARG, "cb_alloc_free_seq: NULL allocator");
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return fail(CB_ERR_INVALID_ARG, "cb_alloc_free_seq: no sequence %d", seq);
  for (int32_t b : it->second.blocks) {
    a->ref[b] -= 1;
    if (a->ref[b] == 0) a->release(b);
  }
  a->seqs.erase(it);
  return CB_OK;
}

int32_t cb_alloc_num_free(const cb_alloc* a) { return a ? a->free_count() : 0; }

cb_status cb_alloc_set_prefix_caching(cb_alloc* a, int32_t enable) {
  if (a == nullptr) return fail(CB_ERR_INVALID_ARG, "cb_alloc_set_prefix_caching: NULL");
  if (!a->seqs.empty())
    return fail(CB_ERR_INVALID_ARG, "cb_alloc_set_prefix_caching: set it before any sequence");
  a->prefix = enable != 0;
  return CB_OK;
}

int32_t cb_alloc_num_cached(const cb_alloc* a) { return a ? (int32_t)a->by_hash.size() : 0; }

cb_status cb_alloc_add_seq_cached(cb_alloc* a, int32_t seq, const int32_t* tokens,
                                  int32_t n_tokens, int32_t* n_cached) {
  if (n_cached != nullptr) *n_cached = 0;
  if (a == nullptr || n_tokens < 1 || tokens == nullptr)
    return fail(CB_ERR_INVALID_ARG, "cb_alloc_add_seq_cached: bad argument");
  if (a->seqs.count(seq))
    return fail(CB_ERR_INVALID_ARG, "cb_alloc_add_seq_cached: sequence %d exists", seq);
  SeqBlocks sq;
  if (a->prefix) {
    // Longest chain of cached full blocks, leaving at least the last token to compute.
    const int32_t full = (n_tokens - 1) / a->bs;
    uint64_t h = 0;
    for (int32_t j = 0; j < full && j < a->max_blocks; ++j) {
      const int32_t* tk = tokens + (size_t)j * a->bs;
      const uint64_t hj = block_hash(h, tk, a->bs);
      auto it = a->by_hash.find(hj);
      if (it == a->by_hash.end()) break;
      const int32_t b = it->second;
      if (a->bparent[b] != h || std::memcmp(a->btokens[b].data(), tk, sizeof(int32_t) * a->bs))
        break;  // a hash collision: not this content
      a->retain(b);
      sq.blocks.push_back(b);
      h = hj;
    }
    sq.len = (int32_t)sq.blocks.size() * a->bs;
    sq.hashed = (int32_t)sq.blocks.size();
    sq.chain = h;
  }
  if (n_cached != nullptr) *n_cached = sq.len;
  a->seqs.emplace(seq, std::move(sq));
  return CB_OK;
}

cb_status cb_alloc_hash_blocks(cb_alloc* a, int32_t seq, const int32_t* tokens, int32_t n_tokens) {
  if (a == nullptr) return fail(CB_ERR_INVALID_ARG, "cb_alloc_hash_blocks: NULL allocator");
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return fail(CB_ERR_INVALID_ARG, "cb_alloc_hash_blocks: no sequence %d", seq);
  if (!a->prefix) return CB_OK;
  SeqBlocks& sq = it->second;
  if (n_tokens > sq.len || (n_tokens > 0 && tokens == nullptr))
    return fail(CB_ERR_INVALID_ARG, "cb_alloc_hash_blocks: %d tokens, sequence holds %d", n_tokens,
                sq.len);
  const int32_t full = n_tokens / a->bs;
  for (int32_t j = sq.hashed; j < full; ++j) {
    const int32_t b = sq.blocks[j];
    const int32_t* tk = tokens + (size_t)j * a->bs;
    const uint64_t hj = block_hash(sq.chain, tk, a->bs);
    if (a->bhash[b] == 0 && a->ref[b] == 1 && !a->by_hash.count(hj)) {
      a->bhash[b] = hj;
      a->bparent[b] = sq.chain;
      a->btokens[b].assign(tk, tk + a->bs);
      a->stamp[b] = a->next_stamp++;
      a->by_hash[hj] = b;
    }
    sq.chain = hj;
    sq.hashed = j + 1;
  }
  return CB_OK;
}

int32_t cb_alloc_ref_count(const cb_alloc* a, int32_t block) {
  if (a == nullptr || block < 0 || block >= a->num_blocks) return -1;
  return a->ref[block];
}

cb_status cb_alloc_table(const cb_alloc* a, int32_t seq, int32_t* blocks, int32_t cap,
                         int32_t* n_blocks, int32_t* n_tokens) {
  if (a == nullptr) return fail(CB_ERR_INVALID_ARG, "cb_alloc_table: NULL allocator");
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return fail(CB_ERR_INVALID_ARG, "cb_alloc_table: no sequence %d", seq);
  const SeqBlocks& sq = it->second;
  const int32_t nb = (int32_t)sq.blocks.size();
  if (blocks != nullptr)
    for (int32_t i = 0; i < nb && i < cap; ++i) blocks[i] = sq.blocks[i];
  if (n_blocks != nullptr) *n_blocks = nb;
  if (n_tokens != nullptr) *n_tokens = sq.len;
  return CB_OK;
}

// ------------------------------------------------------------------------------- scheduler

cb_status cb_sched_create(cb_alloc* alloc, const cb_sched_config* cfg, cb_sched** out) {
  if (out == nullptr) return fail(CB_ERR_INVALID_ARG, "cb_sched_create: out is NULL");
  *out = nullptr;
  if (alloc == nullptr || cfg == nullptr || cfg->max_batch_tokens < 1 ||
      cfg->max_requests_per_batch < 1 ||
      (cfg->policy != CB_SCHED_FIFO && cfg->policy != CB_SCHED_PREFILL_FIRST))
    return fail(CB_ERR_INVALID_ARG, "cb_sched_create: bad configuration");
  cb_sched* s = new (std::nothrow) cb_sched;
  if (s == nullptr) return fail(CB_ERR_INVALID_ARG, "cb_sched_create: out of host memory");
  s->alloc = alloc;
  s->cfg = *cfg;
  *out = s;
  return CB_OK;
}

void cb_sched_destroy(cb_sched* s) { delete s; }

cb_status cb_sched_add_request(cb_sched* s, int32_t id, int32_t prompt_len,
                               int32_t max_new_tokens) {
  if (s == nullptr || prompt_len < 1 || max_new_tokens < 1)
    return fail(CB_ERR_INVALID_ARG, "cb_sched_add_request: bad argument");
  if (s->index.count(id) || s->alloc->seqs.count(id))
    return fail(CB_ERR_INVALID_ARG, "cb_sched_add_request: id %d in use", id);
  const int64_t tokens = (int64_t)prompt_len + max_new_tokens - 1;
  if (cb_alloc::blocks_for(tokens, s->alloc->bs) > s->alloc->max_blocks)
    return fail(CB_ERR_UNSUPPORTED, "cb_sched_add_request: %lld tokens exceed max_blocks_per_seq",
                (long long)tokens);
  cb_sched::Request r;
  r.id = id;
  r.prompt = prompt_len;
  r.max_new = max_new_tokens;
  s->index[id] = s->reqs.size();
  s->reqs.push_back(r);
  return CB_OK;
}

cb_status cb_sched_add_request_tokens(cb_sched* s, int32_t id, const int32_t* tokens,
                                      int32_t prompt_len, int32_t max_new_tokens) {
  if (tokens == nullptr) return fail(CB_ERR_INVALID_ARG, "cb_sched_add_request_tokens: NULL tokens");
  const cb_status st = cb_sched_add_request(s, id, prompt_len, max_new_tokens);
  if (st != CB_OK) return st;
  s->reqs.back().tokens.assign(tokens, tokens + prompt_len);
  return CB_OK;
}

cb_status cb_sched_fork_request(cb_sched* s, int32_t parent, int32_t child,
                                int32_t max_new_tokens) {
  if (s == nullptr) return fail(CB_ERR_INVALID_ARG, "cb_sched_fork_request: NULL scheduler");
  auto it = s->index.find(parent);
  if (it == s->index.end() || s->reqs[it->second].state != cb_sched::kDecode)
    return fail(CB_ERR_INVALID_ARG, "cb_sched_fork_request: parent %d is not decoding", parent);
  if (s->index.count(child) || s->alloc->seqs.count(child))
    return fail(CB_ERR_INVALID_ARG, "cb_sched_fork_request: id %d in use", child);
  const cb_sched::Request p = s->reqs[it->second];
  if (max_new_tokens < p.generated)
    return fail(CB_ERR_INVALID_ARG, "cb_sched_fork_request: max_new_tokens below the parent's %d",
                p.generated);
  const int64_t tokens = (int64_t)p.prompt + max_new_tokens - 1;
  if (cb_alloc::blocks_for(tokens, s->alloc->bs) > s->alloc->max_blocks)
    return fail(CB_ERR_UNSUPPORTED, "cb_sched_fork_request: %lld tokens exceed max_blocks_per_seq",
                (long long)tokens);
  const cb_status st = cb_alloc_fork(s->alloc, parent, child);
  if (st != CB_OK) return st;
  cb_sched::Request c = p;
  c.id = child;
  c.max_new = max_new_tokens;
  s->index[child] = s->reqs.size();
  s->reqs.push_back(c);
  return CB_OK;
}

int32_t cb_sched_num_active(const cb_sched* s) {
  if (s == nullptr) return 0;
  int32_t n = 0;
  for (const auto& r : s->reqs) n += r.state != cb_sched::kDone;
  return n;
}

cb_status cb_sched_step(cb_sched* s, cb_batch* out) {
  if (s == nullptr || out == nullptr || out->seq_ids == nullptr || out->cu_seqlens_q == nullptr ||
      out->kv_lens == nullptr || out->block_table == nullptr ||
      out->cap_seqs < s->cfg.max_requests_per_batch ||
      out->max_blocks < s->alloc->max_blocks ||
      (out->cap_cow > 0 && (out->cow_src == nullptr || out->cow_dst == nullptr)))
    return fail(CB_ERR_INVALID_ARG, "cb_sched_step: output arrays missing or too small");
  cb_alloc* A = s->alloc;
  out->num_seqs = out->num_tokens = out->num_cow = out->num_decode = out->num_finished = 0;
  out->num_cached = 0;
  out->cu_seqlens_q[0] = 0;

  // Retire the requests that produced all their tokens last step.
  for (auto& r : s->reqs) {
    if (r.state != cb_sched::kDone && r.generated >= r.max_new) {
      if (A->seqs.count(r.id)) cb_alloc_free_seq(A, r.id);
      r.state = cb_sched::kDone;
      out->num_finished += 1;
    }
  }

  int32_t budget = s->cfg.max_batch_tokens;
  // Admit `n` tokens of request r; false (nothing changes) when the blocks do not suffice.
  auto admit = [&](cb_sched::Request& r, int32_t n) -> bool {
    if (n <= 0) return false;
    const bool fresh = !A->seqs.count(r.id);
    if (cb_alloc_blocks_needed(A, r.id, n) > A->free_count()) return false;
    if (fresh) {
      if (cb_alloc_add_seq(A, r.id, n) != CB_OK) return false;
    } else {
      int32_t src = -1, dst = -1, nc = 0;
      if (cb_alloc_append(A, r.id, n, &src, &dst, &nc) != CB_OK) return false;
      if (nc) {
        if (out->num_cow >= out->cap_cow) {
          fail(CB_ERR_INVALID_ARG, "cb_sched_step: cap_cow too small");
          return false;
        }
        out->cow_src[out->num_cow] = src;
        out->cow_dst[out->num_cow] = dst;
        out->num_cow += 1;
      }
    }
    const SeqBlocks& sq = A->seqs.at(r.id);
    const int32_t i = out->num_seqs;
    out->seq_ids[i] = r.id;
    out->cu_seqlens_q[i + 1] = out->cu_seqlens_q[i] + n;
    out->kv_lens[i] = sq.len;
    int32_t* row = out->block_table + (size_t)i * out->max_blocks;
    const int32_t nb = (int32_t)sq.blocks.size();
    for (int32_t j = 0; j < out->max_blocks; ++j) row[j] = j < nb ? sq.blocks[j] : -1;
    out->num_seqs += 1;
    out->num_tokens += n;
    budget -= n;
    if (r.state == cb_sched::kDecode) {
      out->num_decode += 1;
      r.generated += 1;
    } else {
      r.done += n;
      r.state = cb_sched::kPrefill;
      if (A->prefix && !r.tokens.empty()) cb_alloc_hash_blocks(A, r.id, r.tokens.data(), r.done);
      if (r.done == r.prompt) {
        r.state = cb_sched::kDecode;
        r.generated = 1;  // the last prompt position gives the first token
      }
    }
    return true;
  };
  // Largest prefix of the remaining prompt (<= budget) whose slots the free blocks and the
  // table width cover: the slack of the last block (after its copy, when it is shared) plus
  // block_size tokens per free block.
  auto fit_chunk = [&](const cb_sched::Request& r) -> int32_t {
    int64_t n = r.prompt - r.done;
    if (n > budget) n = budget;
    int64_t fit;
    auto it = A->seqs.find(r.id);
    const int64_t free_blocks = (int64_t)A->free_count();
    if (it == A->seqs.end()) {
      fit = std::min<int64_t>(free_blocks, A->max_blocks) * A->bs;
    } else {
      const SeqBlocks& sq = it->second;
      const int64_t nb = (int64_t)sq.blocks.size();
      const int64_t slack = nb * A->bs - sq.len;
      const bool cow = slack > 0 && A->ref[sq.blocks.back()] > 1;
      const int64_t spare = free_blocks - (cow ? 1 : 0);
      if (spare < 0) return 0;
      fit = slack + std::min<int64_t>(spare, A->max_blocks - nb) * A->bs;
    }
    return (int32_t)(n < fit ? n : fit);
  };
  const int32_t cap = s->cfg.max_requests_per_batch;
  // Requests that finish their prompt in a pass become decoding; they must not decode in the
  // same step, so each pass only looks at the state requests had when the step started.
  std::vector<cb_sched::State> start(s->reqs.size());
  for (size_t i = 0; i < s->reqs.size(); ++i) start[i] = s->reqs[i].state;
  auto pass_on_start = [&](cb_sched::State want) {
    for (size_t i = 0; i < s->reqs.size(); ++i) {
      if (out->num_seqs >= cap || budget <= 0) return;
      auto& r = s->reqs[i];
      if (start[i] != want || r.state != want) continue;
      if (want == cb_sched::kDecode) {
        if (r.generated < r.max_new) admit(r, 1);
      } else if (want == cb_sched::kWaiting && A->prefix && !r.tokens.empty()) {
        // Prefix caching: start from the longest cached chain of full prompt blocks; the
        // chunk then covers the rest.  Nothing changes if no token of it can be admitted.
        int32_t cached = 0;
        if (cb_alloc_add_seq_cached(A, r.id, r.tokens.data(), r.prompt, &cached) != CB_OK) continue;
        r.done = cached;
        if (admit(r, fit_chunk(r))) {
          out->num_cached += cached;
        } else {
          cb_alloc_free_seq(A, r.id);
          r.done = 0;
        }
      } else {
        admit(r, fit_chunk(r));
      }
    }
  };
  if (s->cfg.policy == CB_SCHED_FIFO) {
    pass_on_start(cb_sched::kDecode);
    pass_on_start(cb_sched::kPrefill);
    pass_on_start(cb_sched::kWaiting);
  } else {
    pass_on_start(cb_sched::kPrefill);
    pass_on_start(cb_sched::kDecode);
    pass_on_start(cb_sched::kWaiting);
  }
  return CB_OK;
}

}  // extern "C"
