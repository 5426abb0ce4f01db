"""Oracle of KV-cache offload / reload and of their FIFO chunk order (test infrastructure only).

Source: "Accelerating Large-Scale Reasoning Model Inference with Sparse
Self-Speculative Decoding" (SparseSpec), MLSys 2026 talk-notes page, section
"Dynamic KV-cache management" (paper Sec. 4.4): instead of predicting output
lengths the scheduler fills GPU memory with KV cache; the cache of requests that
no longer fit is moved to host memory asynchronously, chunk by chunk, and
offloads and loads happen in FIFO order so that no request waits unfairly.

The pages fix no layout and no chunk rule.  Plainest reading, taken here:
  - a transfer copies whole pages verbatim (bf16 bit patterns, nothing is
    computed); the host copy lists the pages in the order given (a request's
    block-table order), each page in the cache's own [Hkv][16][128] layout;
  - reload writes the host copy into whichever physical pages the request is
    given next (distinct pages), leaving every other page as it was;
  - FIFO: requests are served in the order they were queued, each request's
    pages in order, at most max_pages pages per chunk.
"""

from __future__ import annotations

import numpy as np


def offload_pages(cache: np.ndarray, pages, host_init: np.ndarray | None = None) -> np.ndarray:
    """Host copy [n, Hkv, 16, 128] of physical pages ``pages`` of ``cache``
    ([num_pages, Hkv, 16, 128]).  An entry outside [0, num_pages) is not copied:
    its host block keeps ``host_init``'s content (zeros when not given)."""
    pages = np.asarray(pages, dtype=np.int64)
    n = pages.shape[0]
    host = np.zeros((n,) + cache.shape[1:], dtype=cache.dtype) if host_init is None else host_init.copy()
    for i in range(n):
        if 0 <= pages[i] < cache.shape[0]:
            host[i] = cache[pages[i]]
    return host


def reload_pages(cache: np.ndarray, pages, host: np.ndarray) -> np.ndarray:
    """``cache`` after writing host entry i into physical page pages[i] (pages
    distinct; an entry outside [0, num_pages) is skipped)."""
    pages = np.asarray(pages, dtype=np.int64)
    out = cache.copy()
    for i in range(pages.shape[0]):
        if 0 <= pages[i] < cache.shape[0]:
            out[pages[i]] = host[i]
    return out


def fifo_chunks(requests, max_pages: int):
    """Chunks (request, first page, count) for requests [(request, n_pages), ...]
    queued in that order: oldest request first, each request's pages in order, at
    most max_pages per chunk."""
    chunks = []
    for request, n_pages in requests:
        first = 0
        while first < n_pages:
            count = min(max_pages, n_pages - first)
            chunks.append((request, first, count))
            first += count
    return chunks
