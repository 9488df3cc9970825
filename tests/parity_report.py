"""Records the parity errors a GPU test measured (whole-tensor and worst (sequence, head)
slice), keyed by the test's id, into the JSON file named by SALA_PARITY_REPORT. Nothing is
written when that variable is unset."""
import json
import os


def record(res: dict) -> None:
    path = os.environ.get("SALA_PARITY_REPORT")
    if not path:
        return
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    data = {}
    if os.path.exists(path):
        with open(path) as f:
            data = json.load(f)
    prev = data.get(test, {})
    for k, v in res.items():
        prev[k] = max(float(v), prev.get(k, 0.0))
    data[test] = prev
    with open(path, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
