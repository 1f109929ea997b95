"""The oracle and the seeded generator against the stored regression fixture."""
import json
import os

import numpy as np

from tests.golden.make_golden import build

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_matches_stored_fixture():
    with open(os.path.join(HERE, "oracle_small.json")) as f:
        stored = json.load(f)
    now = build()
    assert now["case"] == stored["case"]
    for k, v in stored["inputs_head"].items():
        # generator values are float32-rounded; hosts may differ by one libm ulp
        np.testing.assert_allclose(now["inputs_head"][k], v, rtol=1e-6, err_msg=k)
    for k, v in stored["outputs"].items():
        np.testing.assert_allclose(now["outputs"][k], v, rtol=1e-9, atol=1e-12, err_msg=k)
