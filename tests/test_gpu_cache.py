"""The per-shape workspace and graph cache through the C ABI ("[RFC]: Native
Laya inference with Rust and CUDA #14", "Design": capture per shape, replay,
LRU of at most four shapes and 512 MiB of workspaces).

Checked: a new output buffer for a captured shape re-points the graph's last
launch (no new capture) and leaves the old buffer alone; the LRU bounds hold
after every run of a changing-shape stream, with the evictions an independent
model of the policy predicts; every replay of a shape gives the bytes of its
first run."""
import numpy as np
import pytest

import transformer_encoder_bf16_gb300 as te
from transformer_encoder_bf16_gb300 import synth

from gpu_util import require_gpu, to_bits
from test_gpu_forward import encoder_for

pytestmark = pytest.mark.gpu


def sentinel(torch, shape, dtype):
    return torch.full(shape, 7.0, dtype=dtype, device="cuda")


@pytest.mark.parametrize("name,B,S,lr,fp32", [
    ("reduced", 1, 48, None, False),      # last launch: the split-K residual GEMM
    ("reduced", 3, 40, (9, 40), False),   # last launch: the unpack of packed rows
    ("reduced", 1, 48, None, True),
    ("reduced", 3, 40, (9, 40), True),
    ("full", 1, 464, None, False),
    ("full", 16, 512, (32, 512), False)])
def test_new_output_buffer_retargets_the_graph(name, B, S, lr, fp32):
    torch = require_gpu()
    model = synth.REDUCED if name == "reduced" else synth.FULL
    _, base = encoder_for(model, 0)
    enc = te.Encoder(dict(base.model, out_fp32=int(fp32)), base._weights)
    dtype = torch.float32 if fp32 else torch.bfloat16
    ids, lengths = synth.make_inputs(model, B, S, 21, lr)
    shape = (B, S, model["hidden"])
    a = sentinel(torch, shape, dtype)
    enc.run(ids, lengths, a)
    enc.check()
    st0 = enc.cache_stats()
    assert st0["captures"] == 1 and st0["retargets"] == 0
    ref = a.clone()
    a.fill_(7.0)
    b = sentinel(torch, shape, dtype)
    enc.run(ids, lengths, b)
    enc.check()
    st1 = enc.cache_stats()
    assert st1["captures"] == 1 and st1["retargets"] == 1, st1
    assert torch.equal(b, ref)
    assert torch.all(a == 7.0)            # the first buffer is no longer written
    enc.run(ids, lengths, a)              # and back
    enc.check()
    assert torch.equal(a, ref)
    st2 = enc.cache_stats()
    assert st2["captures"] == 1 and st2["retargets"] == 2, st2
    enc.close()


class LruModel:
    """The eviction policy written out: before allocating a new shape, drop
    least-recently-used shapes while the cache holds max_shapes or the new
    bytes would exceed max_bytes."""

    def __init__(self, max_shapes, max_bytes):
        self.max_shapes, self.max_bytes = max_shapes, max_bytes
        self.resident = {}   # shape -> (bytes, last use)
        self.tick = 0
        self.created = self.evicted = 0

    def use(self, shape, nbytes):
        self.tick += 1
        if shape in self.resident:
            self.resident[shape] = (self.resident[shape][0], self.tick)
            return
        while self.resident and (len(self.resident) >= self.max_shapes or
                                 sum(b for b, _ in self.resident.values()) + nbytes >
                                 self.max_bytes):
            victim = min(self.resident, key=lambda k: self.resident[k][1])
            del self.resident[victim]
            self.evicted += 1
        self.resident[shape] = (nbytes, self.tick)
        self.created += 1


def _stress(enc, model, shapes, order, seed):
    torch = require_gpu()
    st = enc.cache_stats()
    lru = LruModel(st["max_shapes"], st["max_bytes"])
    c0, e0 = st["created"], st["evicted"]
    first = {}
    bufs = {}
    for step, k in enumerate(order):
        B, S = shapes[k]
        lr = (1, S) if B > 1 else None
        ids, lengths = synth.make_inputs(model, B, S, seed + k, lr)
        # two output buffers per shape, alternated: retargets between captures
        pool = bufs.setdefault(k, [torch.empty((B, S, model["hidden"]), dtype=torch.bfloat16,
                                               device="cuda") for _ in range(2)])
        out = pool[step % 2]
        enc.run(ids, lengths, out)
        enc.check()
        got = to_bits(out)
        if k in first:
            for b in range(B):
                L = int(lengths[b])
                np.testing.assert_array_equal(got[b, :L], first[k][b, :L])
        else:
            first[k] = got
        lru.use((B, S), enc.workspace_bytes(B, S))
        st = enc.cache_stats()
        assert st["shapes"] == len(lru.resident), (step, st)
        assert st["shapes"] <= st["max_shapes"] and st["bytes"] <= st["max_bytes"], st
        assert st["bytes"] == sum(b for b, _ in lru.resident.values()), (step, st)
        assert st["created"] - c0 == lru.created and st["evicted"] - e0 == lru.evicted, (step, st)
    return lru


def test_changing_shape_stress_lru_and_replay_bytes():
    model = synth.REDUCED
    _, base = encoder_for(model, 0)
    enc = te.Encoder(base.model, base._weights)
    shapes = [(1, 48), (2, 64), (4, 32), (1, 130), (3, 200), (8, 16), (1, 7)]
    rng = np.random.default_rng(3)
    order = list(rng.integers(0, len(shapes), size=30)) + [0, 1, 2, 3, 0, 4, 5, 6, 0]
    lru = _stress(enc, model, shapes, order, 100)
    st = enc.cache_stats()
    assert lru.evicted > 0 and st["captures"] >= st["created"]
    print(f"\n[cache] {st}")
    enc.close()


def test_byte_bound_evicts_before_the_shape_bound():
    model = synth.FULL
    _, base = encoder_for(model, 4)
    enc = te.Encoder(base.model, base._weights)
    shapes = [(16, 512), (16, 496), (16, 480), (16, 464), (15, 512)]
    sizes = [enc.workspace_bytes(B, S) for B, S in shapes]
    st = enc.cache_stats()
    assert sum(sizes[:4]) > st["max_bytes"]          # four such shapes do not fit
    lru = _stress(enc, model, shapes, [0, 1, 2, 3, 4, 0, 2], 200)
    assert lru.evicted > 0
    st = enc.cache_stats()
    assert st["shapes"] < st["max_shapes"]
    print(f"\n[cache] sizes {sizes} -> {st}")
    enc.close()
