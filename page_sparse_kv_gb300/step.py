"""One decode step launched the way a serving loop launches it, and its CUDA-graph capture.

Stream plumbing only (the work is the library's calls): the step forks a side stream for the
decode append (psk_kv_append_and_summarize) beside score + select on the caller's stream, and the
sparse decode waits for both. The overlap is valid when

  * score + select runs without scores_out, so it does not read the summaries of the
    always-kept pages (the tail page among them), and
  * the append writes one token per sequence, which lands in the tail page;

then nothing the append writes is read before the decode, which runs after the join.
"""
from __future__ import annotations

import torch


class DecodeStep:
    """append, score_select and decode are zero-argument callables that make the library's
    calls on the current torch stream (score_select without scores_out)."""

    def __init__(self, append, score_select, decode):
        self.append, self.score_select, self.decode = append, score_select, decode
        self.side = torch.cuda.Stream()

    def launch(self, pre_main=None, pre_side=None, post=None):
        """Launch one step; pre_main / pre_side run first on their stream (input copies, length
        updates), post runs after the decode on the caller's stream."""
        cur = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(cur)
        self.side.wait_event(fork)
        with torch.cuda.stream(self.side):
            if pre_side is not None:
                pre_side()
            self.append()
            join = torch.cuda.Event()
            join.record(self.side)
        if pre_main is not None:
            pre_main()
        self.score_select()
        cur.wait_event(join)
        self.decode()
        if post is not None:
            post()


def capture(fn) -> torch.cuda.CUDAGraph:
    """A CUDA graph of fn's launches (fn is run once beforehand on a side stream to warm up)."""
    stream = torch.cuda.current_stream()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn()
    stream.wait_stream(side)
    with torch.cuda.graph(g):
        fn()
    return g
