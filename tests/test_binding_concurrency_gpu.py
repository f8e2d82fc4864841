"""Calls from several host threads, each on its own stream: the binding keeps
a workspace per (device, stream, thread) and staging buffers per thread, and
the library serialises the enqueueing of host-input prefills per device, so
concurrent calls give the same bits as the same calls one after another."""
import threading

import pytest
import torch

import gated_deltanet_linear_chunk_gb300 as gdn
from gated_deltanet_linear_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu

N_THREADS, REPEATS = 3, 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _problems(lens_of):
    return [inputs.prefill_inputs(lens_of(i), 2, 6, 128, 128, dtype=torch.bfloat16, seed=50 + i,
                                  initial_state_std=0.02) for i in range(N_THREADS)]


def _run_threads(work):
    errors = []

    def wrap(i):
        try:
            work(i)
        except BaseException as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=wrap, args=(i,)) for i in range(N_THREADS)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    if errors:
        raise errors[0]


def test_device_prefill_from_threads():
    dev = torch.device("cuda")
    ps = _problems(lambda i: [700 + 300 * i, 130])
    args = [[x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta, p.cu_seqlens, p.initial_state)]
            for p in ps]
    ref = []
    for a in args:
        o, f = gdn.gdn_chunk_prefill(*a, output_final_state=True)
        ref.append((o.clone(), f.clone()))
    torch.cuda.synchronize()
    got = [[] for _ in range(N_THREADS)]

    def work(i):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for _ in range(REPEATS):
                o, f = gdn.gdn_chunk_prefill(*args[i], output_final_state=True)
                got[i].append((o, f))
        s.synchronize()

    _run_threads(work)
    for i in range(N_THREADS):
        for o, f in got[i]:
            assert torch.equal(o, ref[i][0]) and torch.equal(f, ref[i][1]), f"thread {i}"


def test_host_prefill_from_threads():
    dev = torch.device("cuda")
    ps = _problems(lambda i: [900 + 200 * i])
    hosts = [[x.pin_memory() for x in (p.q, p.k, p.v, p.g, p.beta)] for p in ps]
    h0 = [p.initial_state.to(dev) for p in ps]

    def one(i):
        T, Hv = ps[i].q.shape[0], ps[i].v.shape[1]
        out = torch.empty((T, Hv, 128), dtype=torch.bfloat16).pin_memory()
        fin = torch.empty((1, Hv, 128, 128), device=dev)
        gdn.gdn_chunk_prefill_host(*hosts[i], out, h0[i], fin, pieces=3)
        return out, fin

    ref = []
    for i in range(N_THREADS):
        o, f = one(i)
        torch.cuda.synchronize()
        ref.append((o.clone(), f.clone()))
    got = [[] for _ in range(N_THREADS)]

    def work(i):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for _ in range(REPEATS):
                got[i].append(one(i))
        s.synchronize()

    _run_threads(work)
    for i in range(N_THREADS):
        for o, f in got[i]:
            assert torch.equal(o, ref[i][0]) and torch.equal(f, ref[i][1]), f"thread {i}"


def test_host_prefill_switching_streams():
    """One thread, alternating streams over the same staging buffers: each
    call is ordered after the previous one."""
    dev = torch.device("cuda")
    p = _problems(lambda i: [1500])[0]
    host = [x.pin_memory() for x in (p.q, p.k, p.v, p.g, p.beta)]
    h0 = p.initial_state.to(dev)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for r in range(6):
        with torch.cuda.stream(streams[r % 2]):
            out = torch.empty((1500, 6, 128), dtype=torch.bfloat16).pin_memory()
            fin = torch.empty((1, 6, 128, 128), device=dev)
            gdn.gdn_chunk_prefill_host(*host, out, h0, fin, pieces=4)
            outs.append((out, fin))
    torch.cuda.synchronize()
    for o, f in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(f, outs[0][1])
