"""The C ABI loads without a GPU, exports every symbol rb.h declares, and rejects bad
arguments on the host before anything is enqueued (no compute calls here)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT, load_golden


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__._build_module().build()
    import ragged_mixed_paged_gb300._binding as b

    return b


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "rb.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    names = set(re.findall(r"\b(rb_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"rb_prepare_inputs", "rb_kv_write", "rb_paged_attention", "rb_gather_rows",
            "rb_pad_for_graph", "rb_paged_attention_workspace_size"} <= set(names)
    raw = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def _declared_param_counts():
    """Parameter count of every function prototype in rb.h (comments stripped)."""
    src = open(os.path.join(ROOT, "include", "rb.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    counts = {}
    for m in re.finditer(r"\b(rb_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", src):
        params = " ".join(m.group(2).split())
        counts[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return counts


def test_binding_signatures_match_the_header(lib):
    """Every function the binding types has the parameter count rb.h declares for it."""
    counts = _declared_param_counts()
    typed = {n: len(getattr(lib.lib, n).argtypes) for n in counts
             if getattr(getattr(lib.lib, n, None), "argtypes", None) is not None}
    assert {"rb_step_host_async", "rb_paged_attention", "rb_prepare_inputs"} <= set(typed)
    for n, k in typed.items():
        assert k == counts[n], (n, k, counts[n])


def test_status_strings(lib):
    assert lib.status_string(0) == "ok"
    assert lib.status_string(5) == "unsupported shape"


def test_pad_for_graph_matches_the_pages(lib):
    g = load_golden("padding_waste.json")
    sizes = g["inputs"]["capture_sizes"]
    for n, padded, _ in g["expected"]["graph_padding"]:
        assert lib.pad_for_graph(sizes, n) == padded
    assert lib.pad_for_graph(sizes, 1) == 1
    assert lib.pad_for_graph(sizes, 256) == 256
    assert lib.pad_for_graph(sizes, 257) == 257        # eager beyond the largest size
    assert lib.pad_for_graph([], 5) == 5
    assert lib.pad_for_graph([4, 2], 3) == -1          # unsorted sizes are rejected
    assert lib.pad_for_graph(sizes, -1) == -1
    import oracle
    for n in range(0, 300):
        assert lib.pad_for_graph(sizes, n) == oracle.pad_for_graph(sizes, n)


def _dims(lib, **kw):
    base = dict(block_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128, max_num_reqs=8,
                max_model_len=4096, max_blocks_per_req=256, num_blocks=1000, null_block=0,
                kernel_blocks_per_manager_block=1)
    base.update(kw)
    return lib.rb_dims(*[base[f] for f, _ in lib.rb_dims._fields_])


FAKE = ctypes.c_void_p(0x100000)  # never dereferenced: every call below fails its host checks
MISALIGNED = ctypes.c_void_p(0x100008)


def test_prepare_inputs_host_checks(lib):
    L = lib.lib
    d = _dims(lib)
    args = [FAKE] * 11 + [None] * 3  # token_table .. scalars, no phase flags; stream follows
    assert L.rb_prepare_inputs(None, 1, 1, 1, 1, *args, None) == 1
    assert L.rb_prepare_inputs(ctypes.byref(d), 9, 9, 9, 9, *args, None) == 2   # > max_num_reqs
    assert L.rb_prepare_inputs(ctypes.byref(d), 2, 1, 2, 2, *args, None) == 1   # R_pad < R
    assert L.rb_prepare_inputs(ctypes.byref(d), 1, 1, 3, 2, *args, None) == 1   # N_pad < N
    assert L.rb_prepare_inputs(ctypes.byref(d), 1, 2, 1, 0, *args, None) == 1   # N_pad = 0
    bad = _dims(lib, null_block=1000)
    assert L.rb_prepare_inputs(ctypes.byref(bad), 1, 1, 1, 1, *args, None) == 1
    nul = [FAKE] * 6 + [None] + [FAKE] * 4 + [None] * 3  # query_start_loc missing
    assert L.rb_prepare_inputs(ctypes.byref(d), 1, 1, 1, 1, *nul, None) == 1
    half = [FAKE] * 11 + [FAKE, FAKE, None]  # one flag output without the other
    assert L.rb_prepare_inputs(ctypes.byref(d), 1, 1, 1, 1, *half, None) == 1
    noprompt = [FAKE] * 11 + [None, FAKE, FAKE]  # flags requested without prompt lengths
    assert L.rb_prepare_inputs(ctypes.byref(d), 1, 1, 1, 1, *noprompt, None) == 1
    # manager-block page tables: pool and null page must be whole manager blocks
    for kw in (dict(kernel_blocks_per_manager_block=3),              # 1000 % 3 != 0
               dict(kernel_blocks_per_manager_block=2, null_block=1),
               dict(kernel_blocks_per_manager_block=65, num_blocks=65 * 16),
               dict(kernel_blocks_per_manager_block=-1)):
        bad = _dims(lib, **kw)
        assert L.rb_prepare_inputs(ctypes.byref(bad), 1, 1, 1, 1, *args, None) == 1, kw
        assert _attn(lib, bad) == 1, kw


def test_kv_write_host_checks(lib):
    L = lib.lib
    d = _dims(lib)
    assert L.rb_kv_write(ctypes.byref(d), 4, None, FAKE, FAKE, FAKE, FAKE, None, None) == 1
    assert L.rb_kv_write(ctypes.byref(d), 4, MISALIGNED, FAKE, FAKE, FAKE, FAKE, None, None) == 1
    assert L.rb_kv_write(ctypes.byref(d), -1, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == 1
    odd = _dims(lib, num_kv_heads=1, head_dim=3)
    assert L.rb_kv_write(ctypes.byref(odd), 4, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == 5
    assert L.rb_kv_write(ctypes.byref(d), 0, None, None, None, None, None, None, None) == 0


def _attn(lib, d, R=2, N=4, Np=4, ws=FAKE, ws_bytes=1 << 30, q=FAKE):
    return lib.lib.rb_paged_attention(ctypes.byref(d), R, N, Np, q, FAKE, FAKE, FAKE, FAKE, FAKE,
                                      ctypes.c_float(0.1), FAKE, ws, ws_bytes, None, None)


def test_paged_attention_host_checks(lib):
    assert _attn(lib, _dims(lib, block_size=8)) == 5
    assert _attn(lib, _dims(lib, head_dim=96)) == 5
    assert _attn(lib, _dims(lib, num_q_heads=30)) == 1
    assert _attn(lib, _dims(lib, num_q_heads=64, num_kv_heads=2)) == 5       # group 32
    assert _attn(lib, _dims(lib), R=9) == 2
    assert _attn(lib, _dims(lib), N=5, Np=4) == 1
    assert _attn(lib, _dims(lib), q=MISALIGNED) == 1
    assert _attn(lib, _dims(lib), ws=ctypes.c_void_p(0x100010)) == 1          # not 256-aligned
    assert _attn(lib, _dims(lib), ws_bytes=16) == 2
    d = _dims(lib)
    need = lib.lib.rb_paged_attention_workspace_size(ctypes.byref(d), 2, 4)
    assert need > 0
    assert _attn(lib, d, ws_bytes=need - 1) == 2
    more = lib.lib.rb_paged_attention_workspace_size(ctypes.byref(d), 200, 4)
    assert more > need
    assert lib.lib.rb_paged_attention_workspace_size(None, 2, 4) == 0
    assert lib.lib.rb_paged_attention_workspace_size(ctypes.byref(d), -1, 4) == 0


def test_gather_rows_host_checks(lib):
    L = lib.lib
    assert L.rb_gather_rows(2, 4095, 8, FAKE, FAKE, FAKE, None, None) == 5
    assert L.rb_gather_rows(2, 4096, 8, None, FAKE, FAKE, None, None) == 1
    assert L.rb_gather_rows(2, 4096, 8, MISALIGNED, FAKE, FAKE, None, None) == 1
    assert L.rb_gather_rows(0, 4096, 8, None, None, None, None, None) == 0
    assert L.rb_gather_rows(-1, 4096, 8, FAKE, FAKE, FAKE, None, None) == 1


def _batch(lib, NR=8, **kw):
    b = lib.rb_batch(NR, 64, 8, 0, *([FAKE.value] * 8))
    for k, v in kw.items():
        setattr(b, k, v)
    return b


def _update(lib, S=2, NN=1, NC=1, **kw):
    u = lib.rb_batch_update(S, NN, NC, 0, *([FAKE.value] * 16))
    for k, v in kw.items():
        setattr(u, k, v)
    return u


def test_batch_update_host_checks(lib):
    L = lib.lib
    n = ctypes.c_size_t(0)
    assert L.rb_batch_update_workspace_size(8, ctypes.byref(n)) == 0 and n.value > 0
    small = n.value
    assert L.rb_batch_update_workspace_size(4096, ctypes.byref(n)) == 0 and n.value > small
    assert L.rb_batch_update_workspace_size(4097, ctypes.byref(n)) == 5
    assert L.rb_batch_update_workspace_size(0, ctypes.byref(n)) == 1
    assert L.rb_batch_update_workspace_size(8, None) == 1

    def call(b, u, ws_bytes=small, num_sched=FAKE, err=FAKE, ws=FAKE):
        return L.rb_batch_apply_update(ctypes.byref(b) if b is not None else None,
                                       ctypes.byref(u) if u is not None else None,
                                       num_sched, None, ws, ws_bytes, err, None)

    assert call(None, _update(lib)) == 1
    assert call(_batch(lib), None) == 1
    assert call(_batch(lib, NR=4097), _update(lib)) == 5
    assert call(_batch(lib, reserved=1), _update(lib)) == 1
    assert call(_batch(lib, d_num_rows=None), _update(lib)) == 1
    assert call(_batch(lib), _update(lib, S=9, NN=1, NC=1)) == 2        # S > max_num_reqs
    assert call(_batch(lib), _update(lib, S=1, NN=2, NC=0)) == 1        # NN > S
    assert call(_batch(lib), _update(lib, S=1, NN=0, NC=2)) == 1        # NC > S
    assert call(_batch(lib), _update(lib, S=-1, NN=0, NC=0)) == 1
    assert call(_batch(lib), _update(lib, d_new_tokens=None)) == 1
    assert call(_batch(lib), _update(lib, d_cached_replace=None)) == 1
    assert call(_batch(lib), _update(lib, d_sched_req_id=None)) == 1
    assert call(_batch(lib), _update(lib), num_sched=None) == 1
    assert call(_batch(lib), _update(lib), err=None) == 1
    assert call(_batch(lib), _update(lib), ws=MISALIGNED) == 1
    assert call(_batch(lib), _update(lib), ws_bytes=small - 1) == 2


def test_cascade_prefix_len_host_rule(lib):
    """The library's host rule equals the oracle's on random batches."""
    import numpy as np

    import oracle

    rng = np.random.default_rng(0)
    for _ in range(200):
        R = int(rng.integers(0, 6))
        c = [int(x) for x in rng.integers(0, 500, size=R)]
        shared, B = int(rng.integers(0, 600)), int(rng.choice([1, 16, 32]))
        assert lib.cascade_prefix_len(shared, c, B) == oracle.cascade_prefix_len(shared, c, B)
    assert lib.cascade_prefix_len(-1, [3], 16) == -1
    assert lib.cascade_prefix_len(10, [3], 0) == -1
    assert lib.cascade_prefix_len(10, [-3], 16) == -1


def test_cascade_attention_host_checks(lib):
    L = lib.lib

    def call(d, P, ws_bytes=1 << 30):
        return L.rb_paged_attention_cascade(ctypes.byref(d), 2, 4, 4, P, FAKE, FAKE, FAKE, FAKE,
                                            FAKE, FAKE, ctypes.c_float(0.1), FAKE, FAKE, ws_bytes,
                                            None, None)

    d = _dims(lib)
    assert call(d, 8) == 1                                  # not a whole page
    assert call(d, 16 * 257) == 1                           # more entries than a row has
    assert call(d, -16) == 1
    assert call(_dims(lib, num_q_heads=64, num_kv_heads=2), 16) == 5   # group 32
    r2 = _dims(lib, kernel_blocks_per_manager_block=2)
    assert call(r2, 16) == 1                                # half a manager block
    need = L.rb_paged_attention_cascade_workspace_size(ctypes.byref(d), 2, 4)
    plain = L.rb_paged_attention_workspace_size(ctypes.byref(d), 2, 4)
    assert need > plain
    assert call(d, 16, ws_bytes=need - 1) == 2


def test_step_host_checks(lib):
    L = lib.lib
    assert L.rb_step(None, None) == 1
    args = lib.rb_step_args()
    assert L.rb_step(ctypes.byref(args), None) == 1            # no dims
    d = _dims(lib)
    args.dims = ctypes.pointer(d)
    args.num_reqs = args.num_reqs_padded = 1
    args.num_tokens = args.num_tokens_padded = 1
    assert L.rb_step(ctypes.byref(args), None) == 1            # no metadata buffers
    none = ctypes.POINTER(ctypes.c_void_p)()
    assert L.rb_step_profiled(None, none, 0, None) == 1
    assert L.rb_step_profiled(ctypes.byref(args), none, 2, None) == 1   # null events array
    assert L.rb_step_profiled(ctypes.byref(args), none, -1, None) == 1
    assert L.rb_step_profiled(ctypes.byref(args), none, 0, None) == 1   # no metadata buffers


def test_step_host_copy_checks(lib):
    """rb_step_host rejects bad copy lists (and rb_step's own bad arguments) before it enqueues
    anything: no GPU is touched."""
    L = lib.lib
    none = ctypes.POINTER(lib.rb_host_copy)()
    assert L.rb_step_host(None, none, 0, none, 0, None) == 1
    args = lib.rb_step_args()
    d = _dims(lib)
    args.dims = ctypes.pointer(d)
    args.num_reqs = args.num_reqs_padded = 1
    args.num_tokens = args.num_tokens_padded = 1
    two = (lib.rb_host_copy * 2)()
    buf = ctypes.create_string_buffer(64)
    addr = ctypes.addressof(buf)
    two[0] = lib.rb_host_copy(addr, addr, 16)
    two[1] = lib.rb_host_copy(None, addr, 16)                # null destination, 16 bytes
    assert L.rb_step_host(ctypes.byref(args), none, -1, none, 0, None) == 1   # negative count
    assert L.rb_step_host(ctypes.byref(args), none, 1, none, 0, None) == 1    # null array
    assert L.rb_step_host(ctypes.byref(args), two, 2, none, 0, None) == 1     # null pointer
    assert L.rb_step_host(ctypes.byref(args), none, 0, two, 2, None) == 1
    two[1] = lib.rb_host_copy(None, None, 0)                 # empty copies need no pointers
    assert L.rb_step_host(ctypes.byref(args), two, 2, two, 2, None) == 1      # no metadata buffers


def test_step_host_async_checks(lib):
    """rb_step_host_async rejects what rb_step_host rejects and null events, before it enqueues
    anything: no GPU is touched."""
    L = lib.lib
    none = ctypes.POINTER(lib.rb_host_copy)()
    ev = ctypes.c_void_p(1)  # never dereferenced: every call below fails its host checks first
    assert L.rb_step_host_async(None, none, 0, none, 0, None, None, None, ev, ev) == 1
    args = lib.rb_step_args()
    d = _dims(lib)
    args.dims = ctypes.pointer(d)
    args.num_reqs = args.num_reqs_padded = 1
    args.num_tokens = args.num_tokens_padded = 1
    assert L.rb_step_host_async(ctypes.byref(args), none, -1, none, 0, None, None, None, ev,
                                ev) == 1                                     # negative count
    assert L.rb_step_host_async(ctypes.byref(args), none, 0, none, 0, None, None, None, None,
                                ev) == 1                                     # null in_done
    assert L.rb_step_host_async(ctypes.byref(args), none, 0, none, 0, None, None, None, ev,
                                None) == 1                                   # null step_done
    assert L.rb_step_host_async(ctypes.byref(args), none, 0, none, 0, None, None, None, ev,
                                ev) == 1                                     # no metadata buffers


def test_wait_limit_hook_checks(lib):
    """The attention wait-limit test hook rejects out-of-range settings and restores defaults
    (host state only; no launch)."""
    L = lib.lib
    assert L.rb_debug_attention_wait_limit(10, 0) == 1             # below 100 us
    assert L.rb_debug_attention_wait_limit(20_000_000_000, 0) == 1  # above 10 s
    assert L.rb_debug_attention_wait_limit(0, 2) == 1
    assert L.rb_debug_attention_wait_limit(5_000_000, 1) == 0
    assert L.rb_debug_attention_wait_limit(0, 0) == 0               # back to the defaults
