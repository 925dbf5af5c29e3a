"""Routines of torch's testing helpers used as independent references.

torch.testing._internal.common_quantized holds torch's own implementations of
the cuBLAS block-scaling-factor layout and of FP4 (E2M1) packing.  Its module
imports test-only packages that are not installed, so the named top-level
functions and constants are compiled from torch's installed source by
themselves.  Tests skip when torch ships none of them.
"""
import ast
import importlib.util

import pytest
import torch

_NS = None


def _load():
    global _NS
    if _NS is not None:
        return _NS
    spec = importlib.util.find_spec("torch.testing._internal.common_quantized")
    if spec is None or spec.origin is None:
        pytest.skip("torch ships no quantisation test helpers")
    with open(spec.origin) as f:
        tree = ast.parse(f.read())
    keep = []
    for node in tree.body:
        if isinstance(node, ast.FunctionDef):
            keep.append(node)
        elif isinstance(node, ast.Assign) and all(isinstance(t, (ast.Name, ast.Tuple)) for t in node.targets):
            keep.append(node)
    ns = {"torch": torch, "Tensor": torch.Tensor}
    for node in keep:  # definitions that need modules not imported here are left out
        try:
            exec(compile(ast.Module(body=[node], type_ignores=[]), spec.origin, "exec"), ns)
        except Exception:
            pass
    _NS = ns
    return ns


def get(name):
    fn = _load().get(name)
    if fn is None:
        pytest.skip(f"torch's helper {name} not found")
    return fn
