// The physical block pool behind the block tables ("From MHA to MLA", section 5: each
// request is divided into logical pages that map to a shared physical pool, so no
// request reserves its maximum context as one dense interval).
//
// A free list of block ids (a stack: the most recently released block is handed out
// first) and a used flag per block, so a double release or a foreign id is refused
// instead of corrupting the pool. Growing a table is all-or-nothing. Host-only; one
// thread at a time per pool.
#include <cstdint>
#include <new>
#include <string>
#include <vector>

#include "pda_internal.h"

using pda::fail;

struct pda_block_pool {
  std::vector<int32_t> free_ids;   // stack; back() is handed out next
  std::vector<uint8_t> used;       // per block
};

namespace {

int64_t pages_for(int64_t len, int32_t page) { return (len + page - 1) / page; }

}  // namespace

extern "C" PDA_API pda_status pda_pool_create(pda_block_pool** pool, int64_t num_blocks) {
  pda::clear_error();
  if (pool == nullptr) return fail(PDA_ERR_INVALID_ARG, "pool output pointer is NULL");
  *pool = nullptr;
  if (num_blocks < 1 || num_blocks > INT32_MAX)
    return fail(PDA_ERR_INVALID_ARG, "num_blocks must be in [1, 2^31 - 1]");
  pda_block_pool* p = new (std::nothrow) pda_block_pool();
  if (p == nullptr) return fail(PDA_ERR_INVALID_ARG, "out of host memory");
  try {
    p->free_ids.resize(size_t(num_blocks));
    p->used.assign(size_t(num_blocks), 0);
  } catch (...) {
    delete p;
    return fail(PDA_ERR_INVALID_ARG, "out of host memory");
  }
  // block 0 is handed out first, then 1, 2, ...
  for (int64_t i = 0; i < num_blocks; ++i) p->free_ids[size_t(i)] = int32_t(num_blocks - 1 - i);
  *pool = p;
  return PDA_OK;
}

extern "C" PDA_API void pda_pool_destroy(pda_block_pool* pool) { delete pool; }

extern "C" PDA_API int64_t pda_pool_num_free(const pda_block_pool* pool) {
  return pool ? int64_t(pool->free_ids.size()) : 0;
}

extern "C" PDA_API pda_status pda_pool_grow(pda_block_pool* pool, int32_t* table_row,
                                            int32_t max_blocks_per_seq, int32_t page_size,
                                            int32_t old_len, int32_t new_len) {
  pda::clear_error();
  if (pool == nullptr || table_row == nullptr)
    return fail(PDA_ERR_INVALID_ARG, "pool and table_row must be non-NULL");
  if (page_size < 1 || max_blocks_per_seq < 1)
    return fail(PDA_ERR_INVALID_ARG, "page_size and max_blocks_per_seq must be >= 1");
  if (old_len < 0 || new_len < old_len)
    return fail(PDA_ERR_INVALID_ARG, "need 0 <= old_len <= new_len");
  const int64_t have = pages_for(old_len, page_size);
  const int64_t want = pages_for(new_len, page_size);
  if (want > max_blocks_per_seq)
    return fail(PDA_ERR_INVALID_ARG, "new_len exceeds max_blocks_per_seq * page_size");
  const int64_t need = want - have;
  if (need > int64_t(pool->free_ids.size()))
    return fail(PDA_ERR_OUT_OF_BLOCKS, "the pool has " + std::to_string(pool->free_ids.size()) +
                                           " free blocks, " + std::to_string(need) + " needed");
  for (int64_t lp = have; lp < want; ++lp) {
    const int32_t id = pool->free_ids.back();
    pool->free_ids.pop_back();
    pool->used[size_t(id)] = 1;
    table_row[lp] = id;
  }
  return PDA_OK;
}

extern "C" PDA_API pda_status pda_pool_release(pda_block_pool* pool, int32_t* table_row,
                                               int32_t page_size, int32_t len) {
  pda::clear_error();
  if (pool == nullptr || (table_row == nullptr && len > 0))
    return fail(PDA_ERR_INVALID_ARG, "pool and table_row must be non-NULL");
  if (page_size < 1 || len < 0)
    return fail(PDA_ERR_INVALID_ARG, "page_size must be >= 1 and len >= 0");
  const int64_t n = pages_for(len, page_size);
  // validate every entry before changing anything (flag 2 marks an id seen in this row)
  std::string why;
  int64_t checked = 0;
  for (; checked < n && why.empty(); ++checked) {
    const int32_t id = table_row[checked];
    if (id < 0 || size_t(id) >= pool->used.size())
      why = "table entry " + std::to_string(checked) + " = " + std::to_string(id) +
            " is not a block of this pool";
    else if (pool->used[size_t(id)] == 0)
      why = "block " + std::to_string(id) + " is not in use";
    else if (pool->used[size_t(id)] == 2)
      why = "block " + std::to_string(id) + " appears twice";
    else
      pool->used[size_t(id)] = 2;
  }
  if (!why.empty()) --checked;   // the failing entry was not marked
  for (int64_t lp = 0; lp < checked; ++lp) pool->used[size_t(table_row[lp])] = 1;
  if (!why.empty()) return fail(PDA_ERR_INVALID_ARG, why);
  // the last page's block is pushed first, so a following grow hands the blocks out
  // again in page order; the released entries become -1 (unused)
  for (int64_t lp = n - 1; lp >= 0; --lp) {
    const int32_t id = table_row[lp];
    pool->used[size_t(id)] = 0;
    pool->free_ids.push_back(id);
    table_row[lp] = -1;
  }
  return PDA_OK;
}
