"""Page-task enumeration for the per-logical-page gather, in plain Python.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "MLA cache gather scheduled per logical page" (prhub.com.cn, vllm PR
#51739), section "实现拆解" item 1 and the GatherPageTask /
map_gather_page_task listing in section "关键源码片段". A task is one logical
page of one request: (req, logical_block, page_token_begin, page_token_end,
output_token_begin), with begin/end relative to the page start (end
exclusive). Tasks are numbered request by request, page by page.

Per request r (T = total_tokens, B = block_size):
  output_begin = min(cu[r], T), output_end = min(cu[r+1], T),
  len = max(output_end - output_begin, 0), start = seq_starts[r] or 0,
  pages = ceil((start + len) / B) - floor(start / B),
and page j of r is logical block floor(start / B) + j, copying the part of
[start, start + len) that falls inside it.

Readings where the page leaves a case open:
- len == 0 gives no page. (The page's formula yields one empty page when
  start is not a multiple of B; it copies nothing, so outputs are the same.)
- A request with len > 0 and a negative start gives no page.
- A request with len > 0 whose output_begin is below an earlier boundary of
  cu_seq_lens (some min(cu[j], T), j < r) or below row 0 gives no page: its
  rows would overlap earlier rows or run out of order (the caller gets a
  flag). A decrease of cu_seq_lens by itself only gives len == 0.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

Task = Tuple[int, int, int, int, int]


def _request_span(cu: Sequence[int], seq_starts: Optional[Sequence[int]], r: int, T: int):
    ob = min(int(cu[r]), T)
    oe = min(int(cu[r + 1]), T)
    length = max(oe - ob, 0)
    start = 0 if seq_starts is None else int(seq_starts[r])
    return ob, length, start


def below_earlier_boundary(cu: Sequence[int], r: int, T: int) -> bool:
    """Whether request r's first output row lies below row 0 or below
    min(cu[j], T) for some j < r."""
    ob = min(int(cu[r]), T)
    return ob < max([0] + [min(int(cu[j]), T) for j in range(r)])


def pages_of_request(cu, seq_starts, r: int, T: int, B: int) -> int:
    ob, length, start = _request_span(cu, seq_starts, r, T)
    if length == 0 or start < 0 or below_earlier_boundary(cu, r, T):
        return 0
    first = start // B
    last_exclusive = -(-(start + length) // B)  # ceil
    return last_exclusive - first


def page_tasks(cu: Sequence[int], seq_starts: Optional[Sequence[int]], num_reqs: int,
               total_tokens: int, block_size: int) -> List[Task]:
    """All tasks, in task-id order, by walking each request's logical pages."""
    B, T = block_size, total_tokens
    tasks: List[Task] = []
    for r in range(num_reqs):
        ob, length, start = _request_span(cu, seq_starts, r, T)
        if length == 0 or start < 0 or below_earlier_boundary(cu, r, T):
            continue
        lb = start // B
        while lb * B < start + length:
            page_begin = lb * B
            copy_begin = max(start, page_begin)
            copy_end = min(start + length, page_begin + B)
            tasks.append((r, lb, copy_begin - page_begin, copy_end - page_begin,
                          ob + copy_begin - start))
            lb += 1
    return tasks


def task_by_scan(task_id: int, cu: Sequence[int], seq_starts: Optional[Sequence[int]],
                 num_reqs: int, total_tokens: int, block_size: int) -> Optional[Task]:
    """One task from its flat id the way the page's mapper finds it: walk the
    requests in order, take away each request's page count from the id until
    the id falls inside a request. Returns None past the last task."""
    B, T = block_size, total_tokens
    rel = task_id
    for r in range(num_reqs):
        n = pages_of_request(cu, seq_starts, r, T, B)
        if rel < n:
            ob, length, start = _request_span(cu, seq_starts, r, T)
            lb = start // B + rel
            page_begin = lb * B
            copy_begin = max(start, page_begin)
            copy_end = min(start + length, page_begin + B)
            return (r, lb, copy_begin - page_begin, copy_end - page_begin, ob + copy_begin - start)
        rel -= n
    return None


def num_tasks(cu, seq_starts, num_reqs: int, total_tokens: int, block_size: int) -> int:
    return sum(pages_of_request(cu, seq_starts, r, total_tokens, block_size) for r in range(num_reqs))
