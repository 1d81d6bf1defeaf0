"""Device timeline of the library's kernels, for the benchmark.

Wraps libsstimeline.so (csrc/timeline.cpp): CUPTI concurrent-kernel activity
records, i.e. the start and end of every kernel on the GPU clock, taken while
a captured CUDA graph replays as it does in the timed region (dependent
launches overlap, nothing is serialised).  ``summarize`` turns the records
of n replays into per-kernel figures:

* span: end - start of a launch (a dependent launch starts early and may
  overlap its predecessor, so spans of one replay can add up to more than
  the replay);
* exclusive time: the part of the replay's busy time first covered by that
  launch (launches in start order; a launch is charged only past the latest
  end before it), so the exclusive times of a replay add up to its busy
  time, never more than the replay.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


def available() -> bool:
    return os.path.exists(os.path.join(_HERE, "libsstimeline.so"))


def _lib():
    global _LIB
    if _LIB is None:
        path = os.path.join(_HERE, "libsstimeline.so")
        if not os.path.exists(path):
            raise RuntimeError("libsstimeline.so is not built (the toolkit has no CUPTI?)")
        l = ctypes.CDLL(path)
        l.sstl_get.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_uint64),
                               ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint32),
                               ctypes.c_char_p, ctypes.c_int]
        _LIB = l
    return _LIB


def kernel_kind(name: str) -> str:
    """Library kernel name (e.g. 'k_head_mma') from a mangled or plain name,
    else the name itself."""
    m = re.search(r"(\d+)(k_[A-Za-z0-9_]+)", name)
    if m:
        return m.group(2)[:int(m.group(1))]
    m = re.search(r"\b(k_[A-Za-z0-9_]+)", name)
    return m.group(1) if m else name


class KernelTimeline:
    """``with KernelTimeline() as tl: ...`` records every kernel run inside;
    ``tl.records`` is then [(kind, start_ns, end_ns)] sorted by start."""

    def __init__(self):
        self.records = []

    def __enter__(self):
        l = _lib()
        l.sstl_clear()
        st = l.sstl_start()
        if st != 0:
            raise RuntimeError(f"CUPTI activity tracing did not start ({st})")
        return self

    def __exit__(self, *exc):
        l = _lib()
        l.sstl_stop()
        recs = []
        a, b, s = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint32()
        name = ctypes.create_string_buffer(1024)
        for i in range(l.sstl_count()):
            if l.sstl_get(i, ctypes.byref(a), ctypes.byref(b), ctypes.byref(s), name, 1024) == 0:
                recs.append((kernel_kind(name.value.decode(errors="replace")), a.value, b.value))
        l.sstl_clear()
        recs.sort(key=lambda r: r[1])
        self.records = recs
        return False


def exclusive_times(launches):
    """[(kind, start, end)] in start order -> exclusive time of each launch
    (see the module docstring) and the union (busy) time."""
    out = []
    cur = None
    for _, s, e in launches:
        lo = s if cur is None else max(s, cur)
        out.append(max(0, e - lo))
        cur = e if cur is None else max(cur, e)
    return out, sum(out)


def summarize(records, per_replay: int, kinds_prefix: str = "k_") -> dict:
    """Per-kernel figures of replays of one captured step.

    records: KernelTimeline.records; per_replay: library launches in one
    replay.  Only kernels whose kind starts with kinds_prefix are used, in
    consecutive groups of per_replay.  Returns {"replays", "busy_us",
    "wall_us", "kernels": {kind: {"launches_per_step", "us_per_launch",
    "exclusive_us_per_step", "share"}}, "replay_records": [...]}.
    """
    lib = [r for r in records if r[0].startswith(kinds_prefix)]
    n = len(lib) // per_replay if per_replay > 0 else 0
    if n == 0:
        return {"replays": 0, "kernels": {}}
    acc = {}
    busy = wall = 0.0
    groups = []
    for i in range(n):
        grp = lib[i * per_replay:(i + 1) * per_replay]
        groups.append(grp)
        excl, union = exclusive_times(grp)
        busy += union
        wall += max(e for _, _, e in grp) - grp[0][1]
        for (kind, s, e), x in zip(grp, excl):
            a = acc.setdefault(kind, [0, 0.0, 0.0])
            a[0] += 1
            a[1] += e - s
            a[2] += x
    tot_excl = sum(a[2] for a in acc.values())
    kernels = {}
    for kind, (cnt, span, excl) in sorted(acc.items(), key=lambda kv: -kv[1][2]):
        kernels[kind] = {"launches_per_step": cnt / n, "us_per_launch": span / cnt / 1e3,
                         "exclusive_us_per_step": excl / n / 1e3,
                         "share": excl / tot_excl if tot_excl else 0.0}
    return {"replays": n, "busy_us": busy / n / 1e3, "wall_us": wall / n / 1e3,
            "kernels": kernels, "replay_records": groups}
