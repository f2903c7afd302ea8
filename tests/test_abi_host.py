"""The C-ABI library builds, loads without a GPU, exports every symbol the header declares,
and rejects bad arguments on the host before touching the device. CPU only."""
import ctypes
import os
import re

import pytest

from speculative_decoding_verification_gqa_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load_library()


def declared_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^SV_API\s+[\w\s\*]*?\b(\w+)\s*\(", txt, re.M)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("spec_verify_attn", "spec_accept", "spec_verify_attn_workspace_size",
              "spec_accept_workspace_size", "sv_workspace_status", "sv_status_string"):
        assert s in syms


def test_exports_every_declared_symbol(lib):
    for s in declared_symbols():
        assert hasattr(lib, s), s
    assert set(api.EXPORTS) <= set(declared_symbols())


def test_status_strings(lib):
    for code in range(9):
        assert lib.sv_status_string(code)
    assert lib.sv_status_string(0) == b"ok"
    assert lib.sv_version() >= 100


def _desc(**kw):
    d = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, max_draft_len=3,
             max_seq_len=100, q_rows=8, kv_rows=208, kv_dtype=0, softmax_scale=0.0)
    d.update(kw)
    return api.AttnDesc(**d)


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: checks fail before any launch


def _attn(lib, desc, **ptrs):
    p = dict(q=FAKE, k=FAKE, v=FAKE, T=FAKE, D=FAKE, sc=None, out=FAKE, ws=FAKE)
    p.update(ptrs)
    return lib.spec_verify_attn(None if desc is None else ctypes.byref(desc), p["q"], p["k"],
                                p["v"], p["T"], p["D"], p["sc"], p["out"], p["ws"], 1 << 30,
                                None)


@pytest.mark.parametrize("bad,status", [
    (dict(num_q_heads=6, num_kv_heads=4), 2),   # Hq % Hkv != 0
    (dict(head_dim=96), 2),
    (dict(max_draft_len=-1), 2),
    (dict(max_draft_len=256), 2),
    (dict(batch=-1), 2),
    (dict(kv_dtype=7), 3),
    (dict(softmax_scale=float("nan")), 2),
    (dict(softmax_scale=-1.0), 2),
    (dict(sliding_window=-1), 2),
    (dict(max_seq_len=2 ** 31 - 1024), 2),
    (dict(kv_rows=2 ** 31), 2),
])
def test_attn_rejects_bad_descriptors(lib, bad, status):
    assert _attn(lib, _desc(**bad)) == status
    assert lib.spec_verify_attn_workspace_size(ctypes.byref(_desc(**bad))) == 0


def test_attn_null_and_alignment(lib):
    assert _attn(lib, None) == 1
    assert _attn(lib, _desc(), q=None) == 1
    assert _attn(lib, _desc(), ws=None) == 1
    assert _attn(lib, _desc(kv_dtype=1)) == 1                 # FP8 needs kv_scale
    assert _attn(lib, _desc(), sc=FAKE) == 2                  # bf16 must not get scales
    assert _attn(lib, _desc(), q=ctypes.c_void_p(0x10008)) == 4
    assert _attn(lib, _desc(), ws=ctypes.c_void_p(0x10010)) == 4
    assert _attn(lib, _desc(batch=0), q=None) == 0            # empty batch: nothing to do


def test_accept_rejects_bad_arguments(lib):
    f = FAKE
    assert lib.spec_accept(2, 3, 100, 5, f, f, f, f, f, None, f, 1 << 20, None) == 3
    assert lib.spec_accept(2, -1, 100, 0, f, f, f, f, f, None, f, 1 << 20, None) == 2
    assert lib.spec_accept(2, 3, 0, 0, f, f, f, f, f, None, f, 1 << 20, None) == 2
    assert lib.spec_accept(2, 3, 100, 0, None, f, f, f, f, None, f, 1 << 20, None) == 1
    assert lib.spec_accept(2, 3, 100, 0, f, None, f, f, f, None, f, 1 << 20, None) == 1
    assert lib.spec_accept(2, 3, 100, 2, ctypes.c_void_p(0x10002), f, f, f, f, None, f,
                           1 << 20, None) == 4
    assert lib.spec_accept(0, 3, 100, 0, None, None, None, None, None, None, None, 0,
                           None) == 0


def test_no_device_means_no_workspace_size(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.spec_verify_attn_workspace_size(ctypes.byref(_desc())) == 0
    assert lib.spec_accept_workspace_size(2, 3, 100) == 0


@pytest.mark.parametrize("ctype,cname", [(api.AttnDesc, "sv_attn_desc"),
                                          (api.PlanInfo, "sv_plan_info")])
def test_struct_layouts_match_the_header(tmp_path, ctype, cname):
    """The ctypes mirrors of the header's structs have the C structs' sizes and field
    offsets (a C program compiled against include/specverify.h prints them)."""
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    fields = [f for f, _ in ctype._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "specverify.h"\n'
                   'int main(void) {\n  printf("%%zu", sizeof(%s));\n' % cname +
                   "".join('  printf(" %%zu", offsetof(%s, %s));\n' % (cname, f) for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(root, "include"), "-o", str(exe), str(src)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    assert got[0] == ctypes.sizeof(ctype)
    assert got[1:] == [getattr(ctype, f).offset for f in fields]


def _paged(lib, desc, nb=64, bs=16, table=FAKE, mb=8, **ptrs):
    p = dict(q=FAKE, k=FAKE, v=FAKE, T=FAKE, D=FAKE, sc=None, out=FAKE, ws=FAKE)
    p.update(ptrs)
    return lib.spec_verify_attn_paged(ctypes.byref(desc), p["q"], p["k"], p["v"], nb, bs, table,
                                      mb, p["T"], p["D"], p["sc"], p["out"], p["ws"], 1 << 30,
                                      None)


@pytest.mark.parametrize("kw,status", [
    (dict(bs=12), 2),            # not a power of two
    (dict(bs=4), 2),             # below 8 positions
    (dict(bs=1 << 17), 2),
    (dict(nb=0), 2),
    (dict(nb=2 ** 31 // 16), 2),  # pool rows beyond 32-bit coordinates
    (dict(mb=0), 2),
    (dict(table=None), 1),
    (dict(table=ctypes.c_void_p(0x10002)), 4),
])
def test_paged_rejects_bad_arguments(lib, kw, status):
    assert _paged(lib, _desc(), **kw) == status


def test_paged_checks_the_descriptor_too(lib):
    assert _paged(lib, _desc(head_dim=96)) == 2
    assert _paged(lib, _desc(), q=None) == 1
    assert _paged(lib, _desc(batch=0), q=None) == 0


def test_unit_cta_policy_setter(lib):
    prev = lib.sv_set_unit_ctas(2)
    assert lib.sv_set_unit_ctas(prev) == 2
    assert lib.sv_set_unit_ctas(-2) == -2
    assert lib.sv_set_unit_ctas(1025) == -2
    assert lib.sv_set_unit_ctas(prev) == prev


def test_launch_failure_hook_arms_and_disarms(lib):
    assert lib.sv_inject_launch_failure(-1) == -1  # nothing pending
    assert lib.sv_inject_launch_failure(2) == -1
    assert lib.sv_inject_launch_failure(0) == 2   # re-armed: the previous arming was pending
    assert lib.sv_inject_launch_failure(-1) == 0  # disarmed
    assert lib.sv_inject_launch_failure(-5) == -1


def _stoch(lib, B=2, md=3, V=100, dt=0, temp=1.0, ws_bytes=256, **ptrs):
    p = dict(t=FAKE, d=FAKE, tok=FAKE, dl=FAKE, ua=FAKE, us=FAKE, al=FAKE, nt=FAKE, ws=FAKE)
    p.update(ptrs)
    lib.spec_accept_stochastic.argtypes = [ctypes.c_int32] * 4 + [ctypes.c_void_p] * 6 + [
        ctypes.c_float] + [ctypes.c_void_p] * 3 + [ctypes.c_size_t, ctypes.c_void_p]
    return lib.spec_accept_stochastic(B, md, V, dt, p["t"], p["d"], p["tok"], p["dl"], p["ua"],
                                      p["us"], temp, p["al"], p["nt"], p["ws"], ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=-1), 2), (dict(md=256), 2), (dict(V=0), 2), (dict(V=(1 << 30) + 1), 2),
    (dict(temp=0.0), 2), (dict(temp=-1.0), 2), (dict(temp=float("inf")), 2),
    (dict(temp=float("nan")), 2), (dict(dt=1), 3),
    (dict(t=None), 1), (dict(us=None), 1), (dict(d=None), 1), (dict(ua=None), 1),
    (dict(tok=None), 1), (dict(ws=None), 1),
    (dict(t=ctypes.c_void_p(0x10001)), 4), (dict(us=ctypes.c_void_p(0x10002)), 4),
    (dict(ws=ctypes.c_void_p(0x10080)), 4), (dict(ws_bytes=255), 5),
    (dict(B=0, t=None), 0),
])
def test_stochastic_accept_rejects_bad_arguments(lib, kw, status):
    assert _stoch(lib, **kw) == status


def test_stochastic_accept_workspace_size(lib):
    lib.spec_accept_stochastic_workspace_size.restype = ctypes.c_size_t
    assert lib.spec_accept_stochastic_workspace_size(4, 0, 100) == 256
    assert lib.spec_accept_stochastic_workspace_size(4, 256, 100) == 0
    assert lib.spec_accept_stochastic_workspace_size(-1, 3, 100) == 0
    # max_draft_len 0: draft logits, tokens and keep draws may be NULL (the next check to
    # fail is the workspace size, before any launch)
    assert _stoch(lib, md=0, d=None, tok=None, ua=None, ws_bytes=0) == 5


def _header_signatures():
    """{name: (return type, [parameter types])} of every SV_API declaration."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", " ", txt, flags=re.S)
    out = {}
    for m in re.finditer(r"SV_API\s+([\w\s\*]+?)\b(\w+)\s*\(([^)]*)\)\s*;", txt):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        types = []
        if params and params != "void":
            for p in params.split(","):
                p = " ".join(p.split())
                types.append("ptr" if "*" in p else p.rsplit(" ", 1)[0].replace("const ", ""))
        out[name] = ("ptr" if "*" in ret else ret.replace("const ", "").strip(), types)
    return out


_CTYPES = {"int32_t": ctypes.c_int32, "int": ctypes.c_int, "int64_t": ctypes.c_int64,
           "size_t": ctypes.c_size_t, "float": ctypes.c_float, "sv_status": ctypes.c_int,
           "void": None}


def test_binding_signatures_match_the_header(lib):
    """Every function the Python binding declares to ctypes has the header's parameter
    count and types (pointers as pointers, each scalar with its exact width)."""
    sigs = _header_signatures()
    checked = 0
    for name, (ret, params) in sigs.items():
        fn = getattr(lib, name)
        if fn.argtypes is None:
            continue
        assert len(fn.argtypes) == len(params), name
        for got, want in zip(fn.argtypes, params):
            if want == "ptr":
                assert got is ctypes.c_void_p or hasattr(got, "_type_") and \
                    issubclass(got, ctypes._Pointer), (name, got)
            else:
                assert ctypes.sizeof(got) == ctypes.sizeof(_CTYPES[want]), (name, got, want)
                assert (got in (ctypes.c_float, ctypes.c_double)) == (want == "float"), name
        if ret != "ptr" and _CTYPES.get(ret) is not None:
            assert ctypes.sizeof(fn.restype) == ctypes.sizeof(_CTYPES[ret]), name
        checked += 1
    assert checked >= 15


def test_empty_draft_arrays_get_a_placeholder_pointer():
    """A batch without drafts passes empty draft arrays; the library still wants a pointer
    when max_draft_len > 0, so the binding passes a small allocation of the same dtype
    (never read). Non-empty arrays pass through unchanged."""
    import torch
    for dt in (torch.int32, torch.float32, torch.bfloat16):
        e = torch.empty(0, dtype=dt)
        p = api._or_placeholder(e)
        assert p.numel() > 0 and p.dtype == dt and p.device == e.device
        full = torch.ones(3, dtype=dt)
        assert api._or_placeholder(full) is full


def test_wait_timeout_hook_arms_and_disarms(lib):
    lib.sv_inject_wait_timeout.argtypes = [ctypes.c_int64]
    assert lib.sv_inject_wait_timeout(0) == 0       # nothing pending
    assert lib.sv_inject_wait_timeout(100000) == 0
    assert lib.sv_inject_wait_timeout(5000) == 1    # re-armed: the previous arming was pending
    assert lib.sv_inject_wait_timeout(-3) == 1      # disarmed
    assert lib.sv_inject_wait_timeout(0) == 0


def test_kv_ring_mode_setter(lib):
    """The ring-layout switch of the bf16 tcgen05 kernel: -1 (by the largest row tile), 0
    (paired stages) or 1 (split rings); anything else is rejected and changes nothing."""
    lib.sv_set_kv_rings.argtypes = [ctypes.c_int]
    lib.sv_set_kv_rings.restype = ctypes.c_int
    assert lib.sv_set_kv_rings(1) == -1   # the default is the automatic choice
    assert lib.sv_set_kv_rings(0) == 1
    assert lib.sv_set_kv_rings(2) == -2
    assert lib.sv_set_kv_rings(-2) == -2
    assert lib.sv_set_kv_rings(-1) == 0
    assert lib.sv_set_kv_rings(-1) == -1
