"""The C-ABI library: it builds, loads, exports every function topo.h
declares, mirrors topo.h's structs, and rejects bad arguments on the host
before launching anything.  No call here touches a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import moe_expert_routing_ids_gb300 as topo
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "topo.h")


@pytest.fixture(scope="module")
def lib():
    from moe_expert_routing_ids_gb300 import build
    if not os.path.exists(topo.LIB_PATH):
        try:
            build.build()
        except (OSError, subprocess.CalledProcessError) as ex:
            pytest.skip(f"cannot build libtopoep here: {ex}")
    return topo.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(topo_[a-z_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(topo.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "probe.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "topo.h"\n'
                   'int main(void){printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(topo_cfg),'
                   ' offsetof(topo_cfg, tok_bytes), offsetof(topo_cfg, c_intra),'
                   ' offsetof(topo_cfg, main_rank), sizeof(topo_plan_t), offsetof(topo_plan_t, stats));'
                   'return 0;}\n')
    exe = tmp_path / "probe"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    try:
        subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, "-o", str(exe), str(src)])
    except (OSError, subprocess.CalledProcessError):
        pytest.skip("no C compiler / CUDA headers")
    got = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    C, P = topo.TopoCfg, topo.TopoPlan
    want = [ctypes.sizeof(C), C.tok_bytes.offset, C.c_intra.offset, C.main_rank.offset,
            ctypes.sizeof(P), P.stats.offset]
    assert got == want


def _cfg(**kw):
    base = dict(T=64, E=8, k=2, R=4, ranks_per_node=2, n_slot=1, tok_bytes=8, expert_bytes=100)
    base.update(kw)
    return topo.make_cfg(**base)


BAD = [dict(R=3), dict(ranks_per_node=3), dict(T=63), dict(E=6), dict(k=0), dict(c_intra=0),
       dict(c_inter=0), dict(n_slot=-1), dict(ranks_per_node=64, R=64, E=64, T=64),
       dict(tok_bytes=1 << 30), dict(expert_bytes=1 << 40), dict(max_refine_iters=-1),
       dict(E=4096, R=4, T=64)]


@pytest.mark.parametrize("bad", BAD)
def test_invalid_configs_are_rejected_on_the_host(lib, bad):
    cfg = _cfg(**bad)
    assert topo.topo_workspace_bytes(cfg, 1, topo.TOPO_CALL_CHAIN) == 0
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_hist(cfg, 1, 1 << 20, 1 << 20, 1 << 20, 1 << 30)
    assert ex.value.code == topo.TOPO_EINVAL


def test_null_and_short_workspace(lib):
    cfg = _cfg()
    need = topo.topo_workspace_bytes(cfg, 2, topo.TOPO_CALL_CHAIN)
    assert need > 256
    dummy = 1 << 20
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_hist(cfg, 2, dummy, None, dummy, need)
    assert ex.value.code == topo.TOPO_EINVAL
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_hist(cfg, 2, dummy, dummy, dummy, need - 1)
    assert ex.value.code == topo.TOPO_ENOSPC
    plan = topo.make_plan(dummy, dummy, dummy, dummy, None)
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_plan(cfg, 2, dummy, plan, dummy, need)
    assert ex.value.code == topo.TOPO_EINVAL
    full = topo.make_plan(dummy, dummy, dummy, dummy, dummy)
    for fn, args in ((topo.topo_plan, (cfg, 2, dummy, full, dummy, need - 1)),
                     (topo.topo_reroute, (cfg, 2, dummy, full, dummy, dummy, need - 1)),
                     (topo.topo_dispatch_layout, (cfg, 2, dummy, full, dummy, dummy, dummy, dummy,
                                                  dummy, need - 1))):
        with pytest.raises(topo.TopoError) as ex:
            fn(*args)
        assert ex.value.code == topo.TOPO_ENOSPC
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_ws_reset(None, 1024)
    assert ex.value.code == topo.TOPO_EINVAL
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_cooccur(2, 10, 0, 2, dummy, dummy, dummy, dummy, 256)
    assert ex.value.code == topo.TOPO_EINVAL
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_cooccur(2, 10, 4, 2, dummy, dummy, dummy, dummy, 255)
    assert ex.value.code == topo.TOPO_ENOSPC


def test_workspace_sizes(lib):
    from moe_expert_routing_ids_gb300 import workloads as W
    for w in W.PLAN_WORKLOADS:
        n = topo.topo_workspace_bytes(topo.make_cfg(**w.plan_cfg), w.n_layers, topo.TOPO_CALL_CHAIN)
        assert 256 < n < (1 << 30)
    assert topo.topo_workspace_bytes(None, 0, topo.TOPO_CALL_COOCCUR) == 256


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert topo.topo_strerror(code) != "unknown error"
    assert topo.topo_strerror(-99) == "unknown error"
