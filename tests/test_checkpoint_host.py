"""Checkpoint and resume of the optimizer state, host side (no GPU): the file
layout the header declares, round trips, loading into another plan over the same
tensors (another bucket size, rank count or mesh), and every refusal."""
import os
import struct

import numpy as np
import pytest
import torch

import gradient_sync_zero_gb300 as dps
from gradient_sync_zero_gb300 import build as dbuild

SIZES = [3, 1000, 65536, 13107, 26214, 4097, 27910, 9000]


@pytest.fixture(scope="module", autouse=True)
def built():
    dbuild.build()


def flat_state(plan, seed):
    """Three fp32 [L] arrays with values at tensor slots and zeros in padding."""
    rng = np.random.default_rng(seed)
    off = plan.tensor_offsets()
    out = []
    for _ in range(3):
        a = torch.zeros(plan.L, dtype=torch.float32)
        for t, s in enumerate(SIZES):
            a[off[t]:off[t] + s] = torch.from_numpy(rng.standard_normal(s).astype(np.float32))
        out.append(a)
    return out


def tensor_order(plan, a):
    off = plan.tensor_offsets()
    return torch.cat([a[off[t]:off[t] + s] for t, s in enumerate(SIZES)])


def fnv_words(data: bytes) -> int:
    pad = (-len(data)) % 8
    w = np.frombuffer(data + b"\0" * pad, dtype="<u8")
    h = 0xcbf29ce484222325
    for x in w.tolist():
        h = ((h ^ x) * 0x100000001b3) & 0xFFFFFFFFFFFFFFFF
    return h


def test_file_layout_and_round_trip(tmp_path):
    plan = dps.Plan(SIZES, 32 * 1024, 4)
    st = flat_state(plan, 1)
    path = str(tmp_path / "a.ckpt")
    dps.dp_checkpoint_save(plan, path, *st, step=7)
    raw = open(path, "rb").read()
    magic, ver, arrays, nt, npar, step, chk, P, R, S, z, cap, z2 = struct.unpack("<8sIIqqqQiiiiqq", raw[:80])
    assert (magic, ver, arrays, nt, npar, step) == (b"DPSYNCK1", 1, 7, len(SIZES), sum(SIZES), 7)
    assert (P, R, S, z, cap, z2) == (4, 1, 4, 0, 32 * 1024, 0)
    assert list(np.frombuffer(raw[80:80 + 8 * nt], "<i8")) == SIZES
    body = np.frombuffer(raw[80 + 8 * nt:], "<f4").reshape(3, npar)
    for i in range(3):
        assert np.array_equal(body[i], tensor_order(plan, st[i]).numpy())
    assert fnv_words(raw[80:]) == chk
    got = [torch.full((plan.L,), 9.0) for _ in range(3)]
    assert dps.dp_checkpoint_load(plan, path, *got) == 7
    for a, b in zip(got, st):
        assert torch.equal(a, b)                      # padding reset to zero as well
    assert not os.path.exists(path + ".tmp")


@pytest.mark.parametrize("cap,P,mesh", [(1 << 20, 8, None), (4096, 2, None), (64 * 1024, 8, (2, 4))])
def test_load_into_another_plan(tmp_path, cap, P, mesh):
    """Elastic restart: the state written under one plan lands element for element
    in a plan with another bucket size, rank count or mesh."""
    a = dps.Plan(SIZES, 32 * 1024, 4)
    st = flat_state(a, 2)
    path = str(tmp_path / "b.ckpt")
    dps.dp_checkpoint_save(a, path, *st, step=3)
    b = dps.Plan(SIZES, cap, P, mesh=mesh)
    got = [torch.full((b.L,), -1.0) for _ in range(3)]
    assert dps.dp_checkpoint_load(b, path, *got) == 3
    pad = torch.ones(b.L, dtype=torch.bool)
    for t, s in enumerate(SIZES):
        pad[b.tensor_offsets()[t]:b.tensor_offsets()[t] + s] = False
    for x, y in zip(got, st):
        assert torch.equal(tensor_order(b, x), tensor_order(a, y))
        assert not x[pad].any()


def test_partial_arrays(tmp_path):
    plan = dps.Plan(SIZES, 32 * 1024, 4)
    st = flat_state(plan, 3)
    path = str(tmp_path / "c.ckpt")
    dps.dp_checkpoint_save(plan, path, master=st[0], v=st[2], step=1)
    got = torch.zeros(plan.L)
    dps.dp_checkpoint_load(plan, path, v=got)         # skip master, read v
    assert torch.equal(got, st[2])
    with pytest.raises(dps.DPError) as e:
        dps.dp_checkpoint_load(plan, path, m=torch.zeros(plan.L))
    assert e.value.code == dps.DP_EINVAL and "no m array" in str(e.value)


def test_refusals(tmp_path):
    plan = dps.Plan(SIZES, 32 * 1024, 4)
    st = flat_state(plan, 4)
    path = str(tmp_path / "d.ckpt")
    dps.dp_checkpoint_save(plan, path, *st, step=2)
    raw = open(path, "rb").read()
    dst = torch.full((plan.L,), 5.0)

    def load_bytes(data, p=plan, arr=None):
        q = str(tmp_path / "x.ckpt")
        open(q, "wb").write(data)
        return dps.dp_checkpoint_load(p, q, master=dst if arr is None else arr)

    with pytest.raises(dps.DPError) as e:                 # not a checkpoint
        load_bytes(b"NOTACKPT" + raw[8:])
    assert e.value.code == dps.DP_EINVAL
    with pytest.raises(dps.DPError) as e:                 # unknown version
        load_bytes(raw[:8] + struct.pack("<I", 2) + raw[12:])
    assert e.value.code == dps.DP_EINVAL
    with pytest.raises(dps.DPError) as e:                 # truncated
        load_bytes(raw[:-4])
    assert e.value.code == dps.DP_EINVAL
    other = dps.Plan(SIZES[:-2] + [27909, 9001], 32 * 1024, 4)   # same total, tensors differ
    d2 = torch.full((other.L,), 5.0)
    with pytest.raises(dps.DPError) as e:
        load_bytes(raw, p=other, arr=d2)
    assert e.value.code == dps.DP_EPLAN and "tensor 6" in str(e.value)
    assert (d2 == 5.0).all()                               # refused before anything is written
    with pytest.raises(dps.DPError) as e:
        load_bytes(raw, p=dps.Plan(SIZES[:-1] + [9001], 32 * 1024, 4), arr=torch.zeros(plan.L + 64))
    assert e.value.code == dps.DP_EPLAN and "parameters" in str(e.value)
    bad = bytearray(raw)
    bad[-3] ^= 0x40                                        # one flipped bit in v
    with pytest.raises(dps.DPError) as e:
        load_bytes(bytes(bad))
    assert e.value.code == dps.DP_EINVAL and "checksum" in str(e.value)
    with pytest.raises(dps.DPError) as e:                  # nothing to save
        dps.dp_checkpoint_save(plan, str(tmp_path / "e.ckpt"))
    assert e.value.code == dps.DP_EINVAL
    with pytest.raises(dps.DPError) as e:                  # unwritable location
        dps.dp_checkpoint_save(plan, str(tmp_path / "no" / "such" / "dir.ckpt"), master=st[0])
    assert e.value.code == dps.DP_EINVAL
    lib = dps.lib()
    assert lib.dp_checkpoint_save(plan.handle, path.encode(), dps._ptr(st[0]), None, None, 0, 8,
                                  None) == dps.DP_EINVAL   # unknown flag
    with pytest.raises(ValueError):
        dps.dp_checkpoint_save(plan, path, master=torch.zeros(plan.L - 1))
