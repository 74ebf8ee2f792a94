"""The C-ABI library loads without a GPU and exports every function the
header declares; the Python binding wraps each under the same name."""
import ctypes

import pytest

from _util import ensure_library, header_functions


@pytest.fixture(scope="module")
def lib():
    return ctypes.CDLL(ensure_library())


def test_header_declares_the_path():
    names = header_functions()
    for n in ("ts_topk", "dsa_plan", "dsa_gather_kv", "dsa_refill_pool", "sfa_mla_decode"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in header_functions():
        assert hasattr(lib, n), n


def test_binding_has_the_same_names():
    import decode_dsa_kv_gb300 as d
    for n in header_functions():
        assert callable(getattr(d, n)), n
        assert n in d.EXPORTS


def test_host_side_validation_without_gpu():
    import decode_dsa_kv_gb300 as d
    from decode_dsa_kv_gb300 import _abi
    # argument checks return before touching a device
    assert d.ts_topk(None, 64, None, 1, 64, 8, None, None, 0, None, 0) == _abi.TS_ERR_INVALID_ARG
    assert d.sfa_mla_decode(None, None, 1, 1, 1, 1.0, None, None, None, 0, None, 0) == \
        _abi.TS_ERR_INVALID_ARG
    assert d.ts_status_string(_abi.TS_ERR_WORKSPACE).startswith("workspace")
    assert d.ts_topk_workspace_size(2, 1000, 16) > 2 * 1000 * 8
    assert d.sfa_workspace_size(1, 128, 2048) >= 4 * 128 * 512 * 4  # 4 chunks of 512 rows


def test_group_step_validation_without_gpu():
    """dsa_group_step refuses a bad descriptor before it enqueues anything."""
    import decode_dsa_kv_gb300 as d
    from decode_dsa_kv_gb300 import _abi
    g = d.DsaGroup()
    q = 1 << 20  # any 16-byte aligned address: nothing is read before the checks pass
    assert d.dsa_group_step(g, None, None) == _abi.TS_ERR_INVALID_ARG       # no q
    assert d.dsa_group_step(g, None, q) == _abi.TS_ERR_INVALID_ARG          # layers = 0
    g.layers = _abi.TS_MAX_LAYERS + 1
    assert d.dsa_group_step(g, q, q) == _abi.TS_ERR_INVALID_ARG
    g.B, g.layers, g.k, g.S, g.W, g.H, g.max_ctx, g.ctx_stride = 2, 4, 16, 8, 4, 128, 64, 64
    assert d.dsa_group_step(g, q, q) == _abi.TS_ERR_INVALID_ARG             # no sync words
    g.sync = q + 2
    assert d.dsa_group_step(g, q, q) == _abi.TS_ERR_INVALID_ARG             # sync misaligned
    g.sync = q
    assert d.dsa_group_step(g, None, q) == _abi.TS_ERR_INVALID_ARG          # no scores, no ids
    assert d.dsa_group_step(g, q, q + 8) == _abi.TS_ERR_INVALID_ARG         # q misaligned
    assert d.dsa_group_step(g, q, q) == _abi.TS_ERR_INVALID_ARG             # null buffers
    assert g.step == 0                                                      # nothing enqueued


def header_struct_fields(name, path=None):
    """(field, C type) of `typedef struct { ... } name;` in the header, in order."""
    import re

    from _util import HEADER
    text = open(path or HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    body = re.search(r"typedef struct \{(.*?)\}\s*" + name + r"\s*;", text, flags=re.S).group(1)
    fields = []
    for decl in body.split(";"):
        decl = " ".join(decl.split())
        if not decl:
            continue
        m = re.match(r"((?:const )?\w+)\s*(.*)", decl)
        base, rest = m.group(1), m.group(2)
        for item in rest.split(","):
            item = item.strip()
            stars = item.count("*")
            fields.append((item.replace("*", "").strip(), base + "*" * stars))
    return fields


def test_binding_descriptor_matches_the_header_field_by_field():
    # the ctypes descriptor must lay out exactly what dsa_group_step reads:
    # the same fields, in the same order, each of the same size
    from decode_dsa_kv_gb300 import _abi
    c_size = {"int": 4, "int64_t": 8, "float": 4, "size_t": 8, "uint32_t": 4}
    header = header_struct_fields("dsa_group")
    binding = _abi.DsaGroup._fields_
    assert [f for f, _ in header] == [f for f, _ in binding]
    for (f, ctype), (_, pytype) in zip(header, binding):
        want = 8 if ctype.endswith("*") or ctype == "cudaStream_t" else c_size[ctype]
        assert ctypes.sizeof(pytype) == want, (f, ctype, pytype)


def header_param_counts(path=None):
    """name -> number of parameters of every function the header declares."""
    import re

    from _util import HEADER
    text = open(path or HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(([^)]*)\)\s*;", text, flags=re.M):
        params = " ".join(m.group(2).split())
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_take_as_many_arguments_as_the_header():
    from decode_dsa_kv_gb300 import _abi
    counts = header_param_counts()
    assert set(counts) == set(header_functions())
    for name, n in counts.items():
        assert len(_abi._SIGS[name][1]) == n, name
