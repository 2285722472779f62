"""Shared test plumbing: host <-> device copies of the numpy storage forms, tolerances."""
import numpy as np
import torch

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def to_device(arr: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Upload a numpy storage array (bf16 as uint16 bits) as a torch tensor of ``dtype``."""
    arr = np.ascontiguousarray(arr)
    if dtype == "bf16":
        return torch.from_numpy(arr.view(np.int16)).to(device).view(torch.bfloat16)
    if dtype == "f16":
        return torch.from_numpy(arr.view(np.int16)).to(device).view(torch.float16)
    return torch.from_numpy(arr).to(device)


def to_host(t: torch.Tensor, dtype: str) -> np.ndarray:
    """Download a tensor back into the numpy storage form (bit-exact)."""
    t = t.detach().contiguous().cpu()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    if dtype == "f16":
        return t.view(torch.int16).numpy().view(np.float16)
    return t.numpy()


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_decode_close(got: np.ndarray, ref: np.ndarray, dtype: str) -> None:
    """Tolerance of the decode output against the fp64 oracle.

    fp32 inputs: max abs error <= 1e-5.  bf16/fp16 inputs (fp32 accumulation):
    |err| <= 2e-2 + 1e-2 * |ref| elementwise ("2e-2 absolute and 1e-2
    relative", read in the allclose form).
    """
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), "non-finite output"
    err = np.abs(got - ref)
    if dtype == "f32":
        bound = np.full_like(ref, 1e-5)
    else:
        bound = 2e-2 + 1e-2 * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{int(bad.sum())} elements out of tolerance; worst at {idx}: "
                             f"got {got[idx]!r} ref {ref[idx]!r} err {err[idx]:.3e} bound {bound[idx]:.3e}")


def slots_of(block_tables, seq_ids, positions, block_size) -> np.ndarray:
    """Input construction: the linear slot of logical position ``pos`` of each sequence."""
    return np.array([int(block_tables[b][p // block_size]) * block_size + p % block_size
                     for b, p in zip(seq_ids, positions)], dtype=np.int64)
