"""Independent calls that overlap on the GPU: the no-sync route, the dispatch
and the combine of two different problems (axolotl torch_dispatch,
compute_send_counts / build_send_layout / dispatch / combine, with NeMo
uccl_ep.buffer Buffer.dispatch worst-case sizing), each with its own
workspace, error word and outputs, enqueued interleaved on two streams and
from two host threads.  Nothing is shared between the calls but the library,
so each must match the oracle exactly as if it ran alone."""
import threading

import numpy as np
import torch
import pytest

import combine_send_counts_gb300 as ep
import oracle
from _paths import assert_equal, bits16, np_, randn_bf16, routing_inputs

pytestmark = pytest.mark.gpu

PROBLEMS = [
    # T, H, K, E, P, seed
    (3000, 1024, 8, 64, 8, 11),
    (5000, 2048, 6, 96, 4, 12),
]


class _Problem:
    def __init__(self, T, H, K, E, P, seed):
        self.T, self.H, self.K, self.E, self.P = T, H, K, E, P
        self.El = E // P
        self.x = randn_bf16(T, H, seed)
        self.idx, self.w = routing_inputs(T, K, E, seed + 1, 0.1)
        lay = oracle.send_path(self.x, self.idx, self.w, None, P, self.El)["layout"]
        self.N = int(lay["n"])
        self.y = randn_bf16(self.N, H, seed + 2)     # the expert outputs of the N rows
        self.want = oracle.send_path(self.x, self.idx, self.w, self.y, P, self.El)
        self.xd, self.idd, self.wd = self.x.cuda(), self.idx.cuda(), self.w.cuda()
        self.W = T * min(K, P)
        self.yd = torch.zeros((self.W, H), dtype=torch.bfloat16, device="cuda")
        self.yd[:self.N].copy_(self.y.cuda())
        self.ws = ep.workspace(T, K, P, self.El)
        self.cws = ep.combine_ws()
        self.err = ep.error_word()
        self.stream = torch.cuda.Stream()
        torch.cuda.synchronize()

    def enqueue(self):
        s = self.stream
        with torch.cuda.stream(s):
            r = ep.route_nosync(self.idd, self.wd, self.P, self.El, self.W, ws=self.ws, err=self.err, stream=s)
            recv = ep.dispatch_rows(self.xd, r["token_pos"], self.W, err=self.err, stream=s)
            out = ep.combine_rows(self.yd, r["token_pos"], err=self.err, stream=s, ws=self.cws)
        return r, recv, out

    def check(self, r, recv, out):
        assert int(self.err.item()) == 0
        lay = self.want["layout"]
        assert int(r["rank_offsets"][self.P].item()) == self.N
        for k in ("token_pos", "send_idx"):
            assert_equal(k, np_(r[k])[: lay[k].shape[0]], lay[k])
        assert_equal("send_token_idx", np_(r["send_token_idx"])[: self.N], lay["send_token_idx"])
        assert_equal("recv_x", bits16(recv[: self.N]), self.want["recv_x"])
        assert_equal("combine", bits16(out), self.want["out"])


def test_two_problems_interleaved_on_two_streams():
    probs = [_Problem(*p) for p in PROBLEMS]
    last = [None] * len(probs)
    for _ in range(3):                      # every call of one problem overlaps the other's
        for i, p in enumerate(probs):
            last[i] = p.enqueue()
    torch.cuda.synchronize()
    for p, res in zip(probs, last):
        p.check(*res)


def test_two_problems_from_two_host_threads():
    probs = [_Problem(*p) for p in PROBLEMS]
    results, errors = [None] * len(probs), []

    def run(i):
        try:
            p = probs[i]
            torch.cuda.set_device(0)
            for _ in range(5):
                results[i] = p.enqueue()
            p.stream.synchronize()
        except Exception as e:   # re-raised in the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(len(probs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a thread did not finish"
    assert not errors, errors
    torch.cuda.synchronize()
    for p, res in zip(probs, results):
        p.check(*res)
