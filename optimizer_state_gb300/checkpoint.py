"""Per-rank shard-set checkpoints of one layer's ZeRO-3 state.

"ZeRO Stages: Sharding Optimizer State, Gradients, and Parameters", "Where
the shards live and what happens on failure": a checkpoint is either a
gathered copy or a per-rank shard set with enough metadata to rebuild the
partitioning; loading it at a different P is a reshuffle (here the device
kernel ``z3_reshard``), and the safe point is between steps.

Format (directory):
  meta.json        layout (n_p list, N, S), step, buffer order, per-file sha256
  rank%05d.bin     rank r's slices, back to back: bf16 shards [S], then fp32
                   master [S], m [S], v [S]   (16 - 2 = 14 bytes per element)

``save`` synchronises the device before copying (the caller must be between
steps).  ``load`` verifies every rank file is present and intact -- a missing
file is a lost rank, reported by number -- and reshards on the device when the
requested rank count differs from the saved one.  ``save_model`` /
``load_model`` do the same for every unit of a multi-unit model, one shard set
per unit, and rebuild resident copies from the loaded shards.
"""
from __future__ import annotations

import hashlib
import json
import os

import numpy as np

FORMAT = "z3-shards-v1"
BUFFERS = (("shards", np.uint16), ("master", np.float32), ("m", np.float32), ("v", np.float32))


class CheckpointError(RuntimeError):
    pass


def _sha256(path: str) -> str:
    h = hashlib.sha256()
    with open(path, "rb") as f:
        for chunk in iter(lambda: f.read(1 << 24), b""):
            h.update(chunk)
    return h.hexdigest()


def rank_file(r: int) -> str:
    return f"rank{r:05d}.bin"


def write_host(path: str, numel, n_ranks: int, S: int, step: int, arrays: dict):
    """Write host arrays (each [N*S], rank-major) as a per-rank shard set."""
    os.makedirs(path, exist_ok=True)
    files = {}
    for r in range(n_ranks):
        fn = rank_file(r)
        with open(os.path.join(path, fn), "wb") as f:
            for name, dt in BUFFERS:
                a = np.ascontiguousarray(arrays[name], dtype=dt).reshape(-1)
                if a.size != n_ranks * S:
                    raise CheckpointError(f"{name}: expected {n_ranks * S} elements, got {a.size}")
                f.write(a[r * S:(r + 1) * S].tobytes())
        files[fn] = _sha256(os.path.join(path, fn))
    meta = {"format": FORMAT, "numel": [int(n) for n in numel], "n_ranks": int(n_ranks),
            "S": int(S), "step": int(step), "buffers": [b for b, _ in BUFFERS], "files": files}
    with open(os.path.join(path, "meta.json"), "w") as f:
        json.dump(meta, f, indent=1)


def read_host(path: str):
    """Read a shard set back: (meta, arrays as in write_host)."""
    try:
        with open(os.path.join(path, "meta.json")) as f:
            meta = json.load(f)
    except OSError as e:
        raise CheckpointError(f"no checkpoint metadata in {path}: {e}") from e
    if meta.get("format") != FORMAT:
        raise CheckpointError(f"unknown checkpoint format {meta.get('format')!r}")
    N, S = meta["n_ranks"], meta["S"]
    missing = [r for r in range(N) if not os.path.exists(os.path.join(path, rank_file(r)))]
    if missing:
        raise CheckpointError(f"rank shard file(s) missing for rank(s) {missing}: the slices "
                              "those ranks owned are lost")
    arrays = {name: np.empty(N * S, dt) for name, dt in BUFFERS}
    for r in range(N):
        fp = os.path.join(path, rank_file(r))
        if _sha256(fp) != meta["files"][rank_file(r)]:
            raise CheckpointError(f"rank {r}: shard file checksum mismatch")
        raw = open(fp, "rb").read()
        off = 0
        for name, dt in BUFFERS:
            n = S * np.dtype(dt).itemsize
            if off + n > len(raw):
                raise CheckpointError(f"rank {r}: shard file truncated")
            arrays[name][r * S:(r + 1) * S] = np.frombuffer(raw[off:off + n], dt)
            off += n
        if off != len(raw):
            raise CheckpointError(f"rank {r}: shard file has trailing bytes")
    return meta, arrays


def save(path: str, layout, shards, master, m, v, step: int):
    """Save device state ([N][S] tensors of ``layout``) between steps."""
    import torch
    torch.cuda.synchronize()

    def host(t, dt):
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        return t.detach().cpu().numpy().view(dt)
    arrays = {"shards": host(shards, np.uint16), "master": host(master, np.float32),
              "m": host(m, np.float32), "v": host(v, np.float32)}
    write_host(path, layout.numel, layout.n_ranks, layout.S, step, arrays)


def load(path: str, n_ranks: int | None = None, device="cuda"):
    """Load a shard set onto the device, resharded to ``n_ranks`` (default:
    the saved rank count).  Returns (layout, dict of [N][S] tensors, step)."""
    import torch

    from . import z3
    meta, arrays = read_host(path)
    src = z3.Layout(meta["numel"], meta["n_ranks"])
    if src.S != meta["S"]:
        raise CheckpointError("metadata S does not match the layout of its parameter list")

    def dev(name, a):
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(device)
        return t.view(torch.bfloat16) if name == "shards" else t
    tensors = {name: dev(name, a) for name, a in arrays.items()}
    if n_ranks is None or n_ranks == meta["n_ranks"]:
        return src, tensors, meta["step"]
    dst = z3.Layout(meta["numel"], n_ranks)
    out = {}
    for name, t in tensors.items():
        o = torch.empty(dst.psi_padded, dtype=t.dtype, device=device)
        z3.z3_reshard(src, dst, t, o)
        out[name] = o
    torch.cuda.synchronize()
    return dst, out, meta["step"]


MODEL_FORMAT = "z3-model-v1"


def save_model(path: str, model):
    """Save every unit of a multi-unit model (``schedule.Model``) between
    steps: one per-rank shard set per unit under ``unit%03d/`` and a
    ``model.json`` with the units' names, parameter counts, resident flags and
    the step counter.  A resident unit's gathered copy is not saved: it is a
    function of the shards."""
    os.makedirs(path, exist_ok=True)
    units = []
    for i, u in enumerate(model.units):
        sub = f"unit{i:03d}"
        save(os.path.join(path, sub), u.L, u.shards, u.master, u.m, u.v, model.t)
        units.append({"dir": sub, "name": u.w.name, "numel": [int(n) for n in u.L.numel],
                      "resident": u.resident is not None})
    with open(os.path.join(path, "model.json"), "w") as f:
        json.dump({"format": MODEL_FORMAT, "step": int(model.t), "units": units}, f, indent=1)


def load_model(path: str, model):
    """Load a saved model into ``model``, whose units must hold the same
    parameters in the same order (each unit may use another rank count: its
    state is resharded on the device).  Resident copies are gathered again
    from the loaded shards, and the model's step counter is restored."""
    import torch

    from . import z3
    try:
        with open(os.path.join(path, "model.json")) as f:
            meta = json.load(f)
    except OSError as e:
        raise CheckpointError(f"no model metadata in {path}: {e}") from e
    if meta.get("format") != MODEL_FORMAT:
        raise CheckpointError(f"unknown model checkpoint format {meta.get('format')!r}")
    if len(meta["units"]) != len(model.units):
        raise CheckpointError(f"checkpoint has {len(meta['units'])} units, the model "
                              f"{len(model.units)}")
    for i, (m, u) in enumerate(zip(meta["units"], model.units)):
        if m["numel"] != [int(n) for n in u.L.numel]:
            raise CheckpointError(f"unit {i}: the saved parameters differ from the model's")
        L, tensors, _ = load(os.path.join(path, m["dir"]), n_ranks=u.L.n_ranks,
                             device=u.shards.device)
        for name in ("shards", "master", "m", "v"):
            getattr(u, name).copy_(tensors[name])
        if u.resident is not None:
            z3.z3_allgather(u.L, u.shards, u.resident)
    model.t = int(meta["step"])
    torch.cuda.synchronize()
