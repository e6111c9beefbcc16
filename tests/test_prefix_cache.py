"""Prefix caching in the native planner, against hotelren.com/news/6181127 §4.3: exact
token-id prefix matching, reuse of the cached K/V pages with positions continuing after the
prefix, block-granular memory, and least-recently-used eviction by block.  Host code only."""
import numpy as np
import pytest

from paged_kv_cache_token_gb300 import binding, build
from paged_kv_cache_token_gb300.native_scheduler import NativeScheduler


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def planner(pages=64, budget=4096):
    return NativeScheduler([], np.arange(pages, dtype=np.int32), budget)


def prompt(n, seed=0):
    return np.random.default_rng(seed).integers(0, 32000, n).astype(np.int32)


def test_second_request_reuses_full_prompt_blocks():
    s = planner()
    a = prompt(100)
    assert s.add_prompt(0, a, 2) == 0            # nothing cached yet
    p = s.next_step()                            # A's whole prompt in one step
    assert list(p.q_lens) == [100] and list(p.context_lens) == [0]
    a_pages = list(p.block_table[0][:7])
    assert s.cached_blocks == 6                  # 6 full blocks (96 tokens); block 7 partial
    # same prompt: 96 tokens reused, the request continues at position 96
    assert s.add_prompt(1, a, 2) == 96
    p = s.next_step()
    i = list(p.rids).index(1)
    assert p.context_lens[i] == 96 and p.q_lens[i] == 4
    assert list(p.block_table[i][:6]) == a_pages[:6]
    assert p.block_table[i][6] not in a_pages    # its own page for tokens 96..99


def test_match_is_exact_and_stops_at_first_differing_block():
    s = planner()
    a = prompt(200)
    s.add_prompt(0, a, 0)
    s.next_step()
    b = a.copy()
    b[50] += 1                                   # block 3 (tokens 48..63) differs
    assert s.add_prompt(1, b, 0) == 48
    c = a.copy()
    c[0] += 1                                    # first block differs: nothing shared
    assert s.add_prompt(2, c, 0) == 0
    d = np.concatenate([a[:64], prompt(30, 1)])  # shares 4 whole blocks, then diverges
    assert s.add_prompt(3, d, 0) == 64


def test_at_least_one_prompt_token_is_left_to_compute():
    s = planner()
    a = prompt(96)                               # exactly 6 blocks
    s.add_prompt(0, a, 0)
    s.next_step()
    assert s.add_prompt(1, a, 1) == 80           # 5 blocks reused, block 6 recomputed
    p = s.next_step()
    assert p.context_lens[0] == 80 and p.q_lens[0] == 16


def test_blocks_register_as_chunks_complete():
    s = NativeScheduler([], np.arange(64, dtype=np.int32), 40)   # 40-token chunks
    a = prompt(100)
    s.add_prompt(0, a, 0)
    s.next_step()                                # tokens 0..39: blocks 0, 1 full
    assert s.cached_blocks == 2
    assert s.add_prompt(1, a, 0) == 32
    s.next_step()                                # A: 40..79 (blocks 2..4); B: 32..71
    assert s.cached_blocks == 5


def test_release_keeps_shared_blocks_cached_and_frees_private_pages():
    s = planner(pages=16)
    a = prompt(40)
    s.add_prompt(0, a, 0)
    s.next_step()
    s.add_prompt(1, a, 0)                        # shares blocks 0, 1
    s.next_step()
    free = s.num_free
    s.release(0)                                 # block 2 of A (partial) was private
    assert s.num_free == free + 1
    assert s.evictable_blocks == 0               # B still holds blocks 0 and 1
    s.release(1)
    assert s.evictable_blocks == 2 and s.cached_blocks == 2
    assert s.add_prompt(2, a, 0) == 32           # still matches after both left
    assert s.evictable_blocks == 0


def test_lru_eviction_by_block_only_when_free_list_is_empty():
    s = planner(pages=8)
    a, b = prompt(40, 1), prompt(40, 2)
    s.add_prompt(0, a, 0)
    s.next_step()                                # pages 0, 1 (shared), 2 (private)
    s.add_prompt(1, b, 0)
    s.next_step()                                # pages 3, 4 (shared), 5 (private)
    s.release(0)                                 # a's blocks unused first ...
    s.release(1)                                 # ... then b's
    assert s.num_free == 4 and s.evictable_blocks == 4
    s.add_prompt(2, prompt(6 * 16, 3), 0)        # 6 pages: 4 free, then evict 2 blocks
    p = s.next_step()
    assert sorted(p.block_table[0][:4]) == [2, 5, 6, 7]     # the free list first
    assert list(p.block_table[0][4:6]) == [0, 1]            # then a's blocks, LRU order
    # b's two blocks stay evictable; the new request registered its own 6 full blocks
    assert s.evictable_blocks == 2 and s.cached_blocks == 8
    assert s.add_prompt(3, a, 0) == 0            # a's blocks are gone ...
    assert s.add_prompt(4, b, 0) == 32           # ... b's survive


def test_referenced_blocks_are_never_evicted():
    s = planner(pages=4)
    a = prompt(40)
    s.add_prompt(0, a, 0)
    s.next_step()                                # pages 0, 1 shared, 2 private; 1 free
    s.add_prompt(1, prompt(40, 9), 0)            # needs 3 pages: 1 free, nothing evictable
    with pytest.raises(binding.PkvError) as e:
        s.next_step()
    assert e.value.status == -7
    assert s.cached_blocks == 2


# ------------------------------------------------------------------ fork + copy-on-write
def test_fork_shares_pages_and_copies_the_partial_page_on_first_write():
    # A's 100-token prompt fills 6 pages and 4 slots of a 7th; B and C fork from it and all
    # three decode: the first two to write into the shared 7th page get copies of it, the
    # last holder writes in place; the full pages stay shared
    s = planner(pages=40)
    s.add_request(0, 0, 100, 3)
    p = s.next_step()
    a_pages = list(p.block_table[0][:7])
    s.fork(0, 1, 3)
    s.fork(0, 2, 3)
    p = s.next_step()
    assert list(p.rids) == [0, 1, 2] and list(p.context_lens) == [100, 100, 100]
    assert p.copies is not None and p.copies.shape == (2, 2)
    assert list(p.copies[:, 0]) == [a_pages[6], a_pages[6]]
    fresh = list(p.copies[:, 1])
    assert len(set(fresh)) == 2 and not set(fresh) & set(a_pages)
    for i in range(3):
        assert list(p.block_table[i][:6]) == a_pages[:6]     # full pages still shared
    assert [p.block_table[i][6] for i in range(3)] == fresh + [a_pages[6]]
    p = s.next_step()                                        # no shared partial page left
    assert p.copies is None


def test_fork_at_a_page_boundary_needs_no_copy_and_release_returns_every_page():
    s = planner(pages=40)
    s.add_request(0, 0, 96, 2)                               # exactly 6 pages
    s.next_step()
    s.fork(0, 1, 2)
    free0 = s.num_free
    p = s.next_step()                                        # both start page 7: fresh pages
    assert p.copies is None
    assert p.block_table[0][6] != p.block_table[1][6]
    assert s.num_free == free0 - 2
    s.next_step()
    assert s.next_step() is None
    s.release(0)                                             # shared pages stay with 1
    assert s.num_free == free0 - 2 + 1
    s.release(1)
    assert s.num_free == 40


def test_fork_release_order_and_copy_capacity():
    s = planner(pages=12)
    s.add_request(0, 0, 40, 1)                               # 2 full pages + 8 slots
    s.next_step()
    for c in (1, 2, 3):
        s.fork(0, c, 1)
    p = s.next_step()                                        # 3 copies of page 3
    assert p.copies.shape == (3, 2)
    assert s.next_step() is None
    for r in (2, 0, 3, 1):
        s.release(r)
    assert s.num_free == 12                                  # every page back exactly once


def test_fork_errors_and_no_pages_leaves_state():
    s = planner(pages=4)
    s.add_request(0, 0, 20, 2)
    with pytest.raises(binding.PkvError):
        s.fork(0, 1, 1)                                      # parent still prefilling
    s.next_step()                                            # 20 tokens: 2 pages
    with pytest.raises(binding.PkvError):
        s.fork(7, 1, 1)                                      # unknown parent
    s.fork(0, 1, 4)
    s.fork(0, 2, 4)
    s.fork(0, 3, 4)
    # 4 requests write into the shared 2nd page: 3 copies, but only 2 pages are free
    with pytest.raises(binding.PkvError):
        s.next_step()
    assert s.num_free == 2                                  # nothing was taken
