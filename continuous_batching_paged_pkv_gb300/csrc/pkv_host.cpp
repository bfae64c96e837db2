// Host side of libpkv: the block pool, step-plan lowering and the attention
// work list. Plain C++; nothing here touches a GPU.
//
// Lucebox, "Continuous batching: Qwen3.8-27B at 301 tok/s across five
// clients, up to 1.97x llama.cpp":
//   §Paged KV and paged attention -- fixed-size blocks in one shared pool,
//     a block table per sequence, finished requests return blocks that a new
//     request can take without moving anyone else;
//   §Admission and step planning are different decisions -- capacity for a
//     request is reserved atomically at admission;
//   §Packing unequal prompt chunks together -- one packed token axis with
//     segment metadata;
//   §Keeping track of each request -- stable slots and a row-to-slot map.
// mlxcel manual, "Continuous batching", §Paged KV cache and prefix sharing --
//   one refcounted, copy-on-write block pool: a request that shares a prompt
//   prefix adopts the donor's blocks by reference instead of prefilling them,
//   and a shared block is copied only when a sequence's contents diverge
//   from it (its first append into that block).
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

constexpr int32_t kVersion = 100;  // 0.1.0

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool supported_block_size(int32_t bs) { return bs == 16 || bs == 32 || bs == 64; }

}  // namespace

struct pkv_pool {
  int64_t num_blocks = 0;
  int32_t block_size = 0, max_slots = 0, max_blocks_per_slot = 0;
  std::vector<int32_t> free_stack;  // top = back()
  std::vector<uint8_t> on_free;     // per block: 1 while on the free stack
  std::vector<int32_t> refs;        // per block: block tables holding it (0 while free)
  std::vector<int32_t> copies;      // pending copy-on-write pairs (source, destination)
  struct Slot {
    bool live = false;
    int64_t length = 0;
    std::vector<int32_t> blocks;
  };
  std::vector<Slot> slots;
};

extern "C" {

const char *pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_OUT_OF_RANGE: return "index out of range";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "buffer too small";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    case PKV_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case PKV_ERR_NO_BLOCKS: return "not enough free KV blocks";
    case PKV_ERR_DEVICE_INDEX: return "device kernel skipped an invalid index";
  }
  return "unknown status";
}

int32_t pkv_version(void) { return kVersion; }

pkv_pool *pkv_pool_create(int64_t num_blocks, int32_t block_size, int32_t max_slots,
                          int32_t max_blocks_per_slot, const int32_t *free_order,
                          int64_t free_order_len) {
  if (num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0 || max_slots <= 0 ||
      max_blocks_per_slot <= 0)
    return nullptr;
  pkv_pool *p = new (std::nothrow) pkv_pool;
  if (!p) return nullptr;
  try {
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->max_slots = max_slots;
    p->max_blocks_per_slot = max_blocks_per_slot;
    p->on_free.assign(static_cast<size_t>(num_blocks), 0);
    p->refs.assign(static_cast<size_t>(num_blocks), 0);
    p->slots.resize(static_cast<size_t>(max_slots));
    if (free_order) {
      if (free_order_len < 0 || free_order_len > num_blocks) {
        delete p;
        return nullptr;
      }
      p->free_stack.reserve(static_cast<size_t>(free_order_len));
      for (int64_t i = 0; i < free_order_len; ++i) {
        int32_t b = free_order[i];
        if (b < 0 || b >= num_blocks || p->on_free[b]) {
          delete p;
          return nullptr;
        }
        p->on_free[b] = 1;
        p->free_stack.push_back(b);
      }
    } else {
      p->free_stack.reserve(static_cast<size_t>(num_blocks));
      for (int64_t b = num_blocks - 1; b >= 0; --b) {
        p->free_stack.push_back(static_cast<int32_t>(b));
        p->on_free[b] = 1;
      }
    }
  } catch (...) {
    delete p;
    return nullptr;
  }
  return p;
}

void pkv_pool_destroy(pkv_pool *pool) { delete pool; }

pkv_status pkv_pool_admit(pkv_pool *p, int32_t slot, int64_t reserve_tokens) {
  if (!p || reserve_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (slot < 0 || slot >= p->max_slots) return PKV_ERR_OUT_OF_RANGE;
  pkv_pool::Slot &s = p->slots[slot];
  if (s.live) return PKV_ERR_INVALID_ARG;
  int64_t need = ceil_div(reserve_tokens, p->block_size);
  if (need > p->max_blocks_per_slot) return PKV_ERR_OUT_OF_RANGE;
  if (need > static_cast<int64_t>(p->free_stack.size())) return PKV_ERR_NO_BLOCKS;
  s.blocks.clear();
  s.blocks.reserve(static_cast<size_t>(p->max_blocks_per_slot));
  for (int64_t i = 0; i < need; ++i) {
    int32_t b = p->free_stack.back();
    p->free_stack.pop_back();
    p->on_free[b] = 0;
    p->refs[b] = 1;
    s.blocks.push_back(b);
  }
  s.live = true;
  s.length = 0;
  return PKV_OK;
}

pkv_status pkv_pool_admit_blocks(pkv_pool *p, int32_t slot, const int32_t *blocks, int32_t num) {
  if (!p || num < 0 || (num > 0 && !blocks)) return PKV_ERR_INVALID_ARG;
  if (slot < 0 || slot >= p->max_slots) return PKV_ERR_OUT_OF_RANGE;
  pkv_pool::Slot &s = p->slots[slot];
  if (s.live) return PKV_ERR_INVALID_ARG;
  if (num > p->max_blocks_per_slot) return PKV_ERR_OUT_OF_RANGE;
  std::vector<uint8_t> seen;
  for (int32_t i = 0; i < num; ++i) {
    int32_t b = blocks[i];
    if (b < 0 || b >= p->num_blocks) return PKV_ERR_OUT_OF_RANGE;
    if (!p->on_free[b]) return PKV_ERR_NO_BLOCKS;  // owned by someone or unavailable
  }
  for (int32_t i = 0; i < num; ++i)
    for (int32_t j = 0; j < i; ++j)
      if (blocks[i] == blocks[j]) return PKV_ERR_INVALID_ARG;
  std::vector<uint8_t> take(static_cast<size_t>(p->num_blocks), 0);
  for (int32_t i = 0; i < num; ++i) take[blocks[i]] = 1;
  std::vector<int32_t> kept;
  kept.reserve(p->free_stack.size());
  for (int32_t b : p->free_stack)
    if (!take[b]) kept.push_back(b);
  p->free_stack.swap(kept);
  s.blocks.assign(blocks, blocks + num);
  for (int32_t i = 0; i < num; ++i) {
    p->on_free[blocks[i]] = 0;
    p->refs[blocks[i]] = 1;
  }
  s.live = true;
  s.length = 0;
  return PKV_OK;
}

pkv_status pkv_pool_release(pkv_pool *p, int32_t slot) {
  if (!p) return PKV_ERR_INVALID_ARG;
  if (slot < 0 || slot >= p->max_slots) return PKV_ERR_OUT_OF_RANGE;
  pkv_pool::Slot &s = p->slots[slot];
  if (!s.live) return PKV_ERR_INVALID_ARG;
  for (auto it = s.blocks.rbegin(); it != s.blocks.rend(); ++it) {
    if (--p->refs[*it] > 0) continue;  // still in another table
    p->free_stack.push_back(*it);
    p->on_free[*it] = 1;
  }
  s.blocks.clear();
  s.live = false;
  s.length = 0;
  return PKV_OK;
}

pkv_status pkv_pool_adopt(pkv_pool *p, int32_t slot, int32_t donor_slot, int64_t num_tokens,
                          int64_t reserve_tokens) {
  if (!p || num_tokens < 0 || reserve_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (slot < 0 || slot >= p->max_slots || donor_slot < 0 || donor_slot >= p->max_slots) return PKV_ERR_OUT_OF_RANGE;
  pkv_pool::Slot &s = p->slots[slot];
  const pkv_pool::Slot &d = p->slots[donor_slot];
  if (s.live || !d.live || slot == donor_slot || num_tokens > d.length) return PKV_ERR_INVALID_ARG;
  const int64_t shared = ceil_div(num_tokens, p->block_size);
  const int64_t total = std::max(shared, ceil_div(reserve_tokens, p->block_size));
  if (total > p->max_blocks_per_slot) return PKV_ERR_OUT_OF_RANGE;
  if (total - shared > static_cast<int64_t>(p->free_stack.size())) return PKV_ERR_NO_BLOCKS;
  s.blocks.assign(d.blocks.begin(), d.blocks.begin() + shared);
  s.blocks.reserve(static_cast<size_t>(p->max_blocks_per_slot));
  for (int64_t i = 0; i < shared; ++i) ++p->refs[s.blocks[i]];
  for (int64_t i = shared; i < total; ++i) {
    int32_t b = p->free_stack.back();
    p->free_stack.pop_back();
    p->on_free[b] = 0;
    p->refs[b] = 1;
    s.blocks.push_back(b);
  }
  s.live = true;
  s.length = num_tokens;
  return PKV_OK;
}

int32_t pkv_pool_block_refs(const pkv_pool *p, int32_t block) {
  if (!p || block < 0 || block >= p->num_blocks) return -1;
  return p->refs[block];
}

pkv_status pkv_pool_take_copies(pkv_pool *p, int32_t *pairs, int64_t capacity, int64_t *num_pairs) {
  if (!p || !num_pairs) return PKV_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(p->copies.size()) / 2;
  *num_pairs = n;
  if (n == 0) return PKV_OK;
  if (!pairs || capacity < n) return PKV_ERR_WORKSPACE_TOO_SMALL;
  std::copy(p->copies.begin(), p->copies.end(), pairs);
  p->copies.clear();
  return PKV_OK;
}

int64_t pkv_pool_slot_length(const pkv_pool *p, int32_t slot) {
  if (!p || slot < 0 || slot >= p->max_slots || !p->slots[slot].live) return -1;
  return p->slots[slot].length;
}

int32_t pkv_pool_slot_blocks(const pkv_pool *p, int32_t slot) {
  if (!p || slot < 0 || slot >= p->max_slots || !p->slots[slot].live) return -1;
  return static_cast<int32_t>(p->slots[slot].blocks.size());
}

pkv_status pkv_pool_get_stats(const pkv_pool *p, pkv_pool_stats *st) {
  if (!p || !st) return PKV_ERR_INVALID_ARG;
  std::memset(st, 0, sizeof(*st));
  st->num_blocks = p->num_blocks;
  st->block_size = p->block_size;
  st->max_slots = p->max_slots;
  st->free_blocks = static_cast<int64_t>(p->free_stack.size());
  for (const auto &s : p->slots) {
    if (!s.live) continue;
    st->live_slots += 1;
    st->live_tokens += s.length;
  }
  for (int32_t r : p->refs) {
    st->owned_blocks += r > 0;
    st->shared_blocks += r > 1;
  }
  return PKV_OK;
}

pkv_status pkv_pool_copy_block_tables(const pkv_pool *p, int32_t *out, int64_t capacity) {
  if (!p || !out) return PKV_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(p->max_slots) * p->max_blocks_per_slot;
  if (capacity < n) return PKV_ERR_WORKSPACE_TOO_SMALL;
  std::fill(out, out + n, -1);
  for (int32_t s = 0; s < p->max_slots; ++s) {
    const auto &b = p->slots[s].blocks;
    std::copy(b.begin(), b.end(), out + static_cast<int64_t>(s) * p->max_blocks_per_slot);
  }
  return PKV_OK;
}

pkv_status pkv_plan_lower(pkv_pool *p, const pkv_segment *plan, int32_t num_segments,
                          int32_t *cu_seqlens_q, int32_t *seq_slot, int32_t *context_lens,
                          int64_t *slot_mapping, int64_t slot_mapping_capacity,
                          int64_t *total_q) {
  if (!p || num_segments < 0 || (num_segments > 0 && !plan) || !cu_seqlens_q ||
      (num_segments > 0 && !seq_slot) || !context_lens || !total_q)
    return PKV_ERR_INVALID_ARG;
  // Validate everything before changing anything.
  std::vector<uint8_t> used(static_cast<size_t>(p->max_slots), 0);
  int64_t rows = 0, new_blocks = 0;
  for (int32_t i = 0; i < num_segments; ++i) {
    const int32_t slot = plan[i].slot, n = plan[i].num_tokens;
    if (slot < 0 || slot >= p->max_slots) return PKV_ERR_OUT_OF_RANGE;
    if (n < 0 || !p->slots[slot].live || used[slot]) return PKV_ERR_INVALID_ARG;
    used[slot] = 1;
    const pkv_pool::Slot &sl = p->slots[slot];
    const int64_t len = sl.length + n;
    const int64_t blocks = ceil_div(len, p->block_size);
    if (blocks > p->max_blocks_per_slot || len > INT32_MAX) return PKV_ERR_OUT_OF_RANGE;
    new_blocks += std::max<int64_t>(0, blocks - static_cast<int64_t>(sl.blocks.size()));
    // The first append lands in block length / block_size; if another table
    // holds that block too, it is copied first (only that block can be shared:
    // adoption shares whole blocks up to the adopted length).
    const int64_t lb0 = sl.length / p->block_size;
    if (n > 0 && lb0 < static_cast<int64_t>(sl.blocks.size()) && p->refs[sl.blocks[lb0]] > 1) ++new_blocks;
    rows += n;
  }
  if (rows > INT32_MAX) return PKV_ERR_OUT_OF_RANGE;
  if (rows > 0 && (!slot_mapping || slot_mapping_capacity < rows))
    return PKV_ERR_WORKSPACE_TOO_SMALL;
  if (new_blocks > static_cast<int64_t>(p->free_stack.size())) return PKV_ERR_NO_BLOCKS;

  int64_t t = 0;
  cu_seqlens_q[0] = 0;
  for (int32_t i = 0; i < num_segments; ++i) {
    pkv_pool::Slot &s = p->slots[plan[i].slot];
    const int32_t n = plan[i].num_tokens;
    const int64_t lb0 = s.length / p->block_size;
    if (n > 0 && lb0 < static_cast<int64_t>(s.blocks.size()) && p->refs[s.blocks[lb0]] > 1) {
      const int32_t old = s.blocks[lb0];
      const int32_t b = p->free_stack.back();
      p->free_stack.pop_back();
      p->on_free[b] = 0;
      p->refs[b] = 1;
      --p->refs[old];
      s.blocks[lb0] = b;
      p->copies.push_back(old);
      p->copies.push_back(b);
    }
    for (int32_t j = 0; j < n; ++j) {
      const int64_t pos = s.length + j;
      const int64_t lb = pos / p->block_size;
      while (static_cast<int64_t>(s.blocks.size()) <= lb) {
        int32_t b = p->free_stack.back();
        p->free_stack.pop_back();
        p->on_free[b] = 0;
        p->refs[b] = 1;
        s.blocks.push_back(b);
      }
      slot_mapping[t++] = static_cast<int64_t>(s.blocks[lb]) * p->block_size + pos % p->block_size;
    }
    s.length += n;
    cu_seqlens_q[i + 1] = static_cast<int32_t>(t);
    seq_slot[i] = plan[i].slot;
  }
  for (int32_t s = 0; s < p->max_slots; ++s)
    context_lens[s] = p->slots[s].live ? static_cast<int32_t>(p->slots[s].length) : 0;
  *total_q = t;
  return PKV_OK;
}

pkv_status pkv_plan_work(const int32_t *cu, int32_t num_seqs, const int32_t *seq_slot,
                         const int32_t *context_lens, int32_t max_slots,
                         int32_t max_blocks_per_slot, int32_t block_size, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t *work,
                         int64_t work_capacity, pkv_work_info *info) {
  if (!info || num_seqs < 0 || !cu || (num_seqs > 0 && (!seq_slot || !context_lens)) ||
      max_slots <= 0 || max_blocks_per_slot <= 0)
    return PKV_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof(*info));
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return PKV_ERR_INVALID_ARG;
  const int32_t group = num_q_heads / num_kv_heads;
  if (group > 16 || (head_dim != 64 && head_dim != 128) || !supported_block_size(block_size))
    return PKV_ERR_UNSUPPORTED;
  if (cu[0] != 0) return PKV_ERR_INVALID_ARG;

  struct Item {
    int32_t w[4];
    int64_t cost;
  };
  std::vector<Item> dec, dec_short, pre, comb, scr;  // dec: full key spans; dec_short: shorter last spans
  int64_t scratch_blocks = 0;
  std::vector<uint8_t> used(static_cast<size_t>(max_slots), 0);
  const int32_t rows_per_tile = 128 / group;
  // Segments of up to 16 / group rows (decode rows and short verify runs) take
  // the split-KV decode path: rows x grouped heads fit its 16 MMA columns.
  const int32_t decode_rows = std::max<int32_t>(1, 16 / group);
  {  // room for every decode span and merge row up front (checked again below)
    int64_t spans = 0, rows = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
      const int32_t n = cu[s + 1] - cu[s], slot = seq_slot[s];
      if (n <= 0 || n > decode_rows || slot < 0 || slot >= max_slots) continue;
      const int64_t sp = ceil_div(std::max<int32_t>(context_lens[slot], 0), PKV_SPLIT_KEYS);
      spans += sp;
      rows += sp > 1 ? n : 0;
    }
    dec.reserve(static_cast<size_t>(std::min<int64_t>(spans, int64_t(1) << 24)));
    comb.reserve(static_cast<size_t>(std::min<int64_t>(rows, int64_t(1) << 24)));
  }
  int32_t partials = 0, rows_max = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t n = cu[s + 1] - cu[s];
    if (n < 0) return PKV_ERR_INVALID_ARG;
    const int32_t slot = seq_slot[s];
    if (slot < 0 || slot >= max_slots) return PKV_ERR_OUT_OF_RANGE;
    if (used[slot]) return PKV_ERR_INVALID_ARG;
    used[slot] = 1;
    const int32_t L = context_lens[slot];
    if (n > L || L < 0) return PKV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(L) > static_cast<int64_t>(max_blocks_per_slot) * block_size)
      return PKV_ERR_OUT_OF_RANGE;
    if (n == 0) continue;
    if (n <= decode_rows) {
      // Partial entry of (span sp, row i): base + sp * n + i. One merge item per
      // row: spans | row << 16 | (n - 1) << 24, and that row's first entry.
      const int32_t spans = static_cast<int32_t>(ceil_div(L, PKV_SPLIT_KEYS));
      if (spans >= (1 << 16)) return PKV_ERR_UNSUPPORTED;
      const int32_t base = spans > 1 ? partials : -1;
      for (int32_t sp = 0; sp < spans; ++sp) {
        const int64_t keys = std::min<int64_t>(PKV_SPLIT_KEYS, L - static_cast<int64_t>(sp) * PKV_SPLIT_KEYS);
        (keys == PKV_SPLIT_KEYS ? dec : dec_short).push_back({{s, slot, sp, base}, keys});
      }
      if (spans > 1) {
        for (int32_t i = 0; i < n; ++i)
          comb.push_back({{s, slot, spans | (i << 16) | ((n - 1) << 24), base + i}, spans});
        partials += spans * n;
      }
      rows_max = std::max(rows_max, n);
    } else {
      // The 8-bit pool's chunk path first widens the segment's whole history
      // into scratch blocks [first, first + blocks) of a bf16 scratch pool.
      const int64_t nblk = ceil_div(L, block_size);
      scr.push_back({{s, slot, static_cast<int32_t>(scratch_blocks), static_cast<int32_t>(nblk)}, 0});
      scratch_blocks += nblk;
      if (scratch_blocks > INT32_MAX) return PKV_ERR_UNSUPPORTED;
      // head_dim 128 runs tiles in pairs on two SMs (the second may be past the segment's end).
      const int32_t tiles = static_cast<int32_t>(ceil_div(n, rows_per_tile));
      const int32_t step = head_dim == 128 ? 2 : 1;
      for (int32_t t = 0; t < tiles; t += step) {
        const int32_t count = std::min(step, tiles - t);
        const int64_t last_row = std::min<int64_t>(n, static_cast<int64_t>(t + count) * rows_per_tile);
        pre.push_back({{s, slot, t, count}, L - n + last_row});
      }
    }
  }
  // Longest first, ties in their original order: the long items start early
  // and the short tails fill in behind them.
  auto by_cost = [](const Item &a, const Item &b) { return a.cost > b.cost; };
  // Full spans all cost the same and are already in order; only the short last spans
  // (one per segment at most) need sorting behind them.
  std::stable_sort(dec_short.begin(), dec_short.end(), by_cost);
  dec.insert(dec.end(), dec_short.begin(), dec_short.end());
  std::stable_sort(pre.begin(), pre.end(), by_cost);
  std::stable_sort(comb.begin(), comb.end(), by_cost);  // long merges start first

  info->num_decode_items = static_cast<int32_t>(dec.size());
  info->num_prefill_items = static_cast<int32_t>(pre.size());
  info->num_combine_items = static_cast<int32_t>(comb.size());
  // merges of more than kLongMergeSpans spans come first (sorted above); the
  // merge launch gives them four lanes per column
  info->num_long_combine_items = static_cast<int32_t>(
      std::count_if(comb.begin(), comb.end(), [](const Item &it) { return it.cost > pkv::kLongMergeSpans; }));
  info->num_partials = partials;
  info->decode_rows_max = rows_max;
  info->num_scratch_items = static_cast<int32_t>(scr.size());
  info->scratch_blocks = scratch_blocks;
  const int64_t items = static_cast<int64_t>(dec.size() + pre.size() + comb.size() + scr.size());
  info->work_words = items * PKV_WORK_WORDS_PER_ITEM;
  auto align256 = [](uint64_t x) { return (x + 255) & ~uint64_t(255); };
  // span partials (sums, then max and denominator), then the decode kernel's task counter
  info->workspace_bytes =
      partials == 0 ? 0
                    : align256(uint64_t(partials) * num_q_heads * head_dim * 4) +
                          align256(uint64_t(partials) * num_q_heads * 2 * 4) + pkv::kCounterBytes;
  info->workspace_bytes_q8 =
      info->workspace_bytes +
      (scratch_blocks == 0 ? 0
                           : 2 * align256(uint64_t(scratch_blocks) * num_kv_heads * block_size * head_dim * 2) +
                                 align256(uint64_t(max_slots) * max_blocks_per_slot * 4));
  if (!work || work_capacity < info->work_words) return PKV_ERR_WORKSPACE_TOO_SMALL;
  int32_t *w = work;
  for (const auto *v : {&dec, &pre, &comb, &scr})
    for (const Item &it : *v) {
      std::memcpy(w, it.w, sizeof(it.w));
      w += PKV_WORK_WORDS_PER_ITEM;
    }
  return PKV_OK;
}

}  // extern "C"
