"""Helpers for GPU tests: moving seeded numpy inputs to the device and outputs back."""
import numpy as np


def to_device(a: np.ndarray):
    """float32 arrays stay float32; uint16 arrays are bf16 bit patterns."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return torch.from_numpy(a).cuda()
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    raise TypeError(a.dtype)


def bits(t) -> np.ndarray:
    """Raw bit patterns of a device tensor (uint32 for float32, uint16 for bf16)."""
    import torch
    if t.dtype == torch.float32:
        return t.contiguous().view(torch.int32).cpu().numpy().view(np.uint32)
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    raise TypeError(t.dtype)


def oracle_bits(v: np.ndarray) -> np.ndarray:
    return v.view(np.uint32) if v.dtype == np.float32 else v.view(np.uint16)


def assert_same(gpu_vals, gpu_idx, ora_vals, ora_idx, what=""):
    """Bit-exact equality of values and indices (tolerance 0)."""
    gi = gpu_idx.cpu().numpy()
    gv = bits(gpu_vals)
    ov = oracle_bits(ora_vals)
    if not np.array_equal(gi, ora_idx):
        bad = np.argwhere(gi != ora_idx)
        first = tuple(bad[0])
        raise AssertionError("%s: index mismatch at %d places, first %s: gpu %d oracle %d"
                             % (what, len(bad), first, gi[first], ora_idx[first]))
    if not np.array_equal(gv, ov):
        bad = np.argwhere(gv != ov)
        raise AssertionError("%s: value bits differ at %d places, first %s" % (what, len(bad), tuple(bad[0])))


def unpack_keys(keys: np.ndarray, ib: int):
    """(value key, position) of composite keys given as raw int64/uint64 bits."""
    u = keys.view(np.uint64)
    mask = np.uint64((1 << ib) - 1)
    return (u >> np.uint64(ib)), (mask - (u & mask)).astype(np.int64)
